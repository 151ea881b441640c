// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "c2kv.h"

namespace c2kv {

constexpr int kMaxDocsPerCompose = 512;   // documents in one c2kv_compose call
constexpr int kMaxBatch = 16;             // sequences in one attention call
constexpr int kMaxHalfDim = 64;           // head_dim <= 128
constexpr int kMaxSplits = 256;           // split-K partitions per (sequence, token, head)

// Device error word bits (see c2kv_device_error).
constexpr unsigned kErrTimeout = 1u;      // a bounded mbarrier wait expired
constexpr unsigned kErrLength = 2u;       // a device-side length exceeded cap / max_keys

// One-time host setup of a kernel (function attributes) and the cluster
// occupancy answers that depend on it.  Attributes belong to the device that
// was current when they were set, so every device has its own entry; `mu`
// makes first use from several host threads safe.
constexpr int kMaxSetupDevices = 64;
struct KernelSetup {
  std::mutex mu;
  int state[kMaxSetupDevices] = {};          // 0 not yet, 1 ready, else -(cudaError_t)
  int clusters[kMaxSetupDevices][17] = {};   // active clusters per size: 0 unknown, -1 none
};

// The current device as an index into KernelSetup (-1 if there is none).
inline int setup_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return d >= 0 && d < kMaxSetupDevices ? d : -1;
}

// Bounded waits give up after this many SM cycles (about 2 s at 2 GHz).
constexpr long long kWaitCycles = 4000000000LL;
constexpr long long kInjectWaitCycles = 1000000LL;   // the test hook's wait (~0.5 ms)

// ---------------------------------------------------------------- RoPE angles
// The angle pos * inv_freq is formed in fp64 and reduced modulo 2*pi with a
// two-constant Cody-Waite reduction (2*pi split into its fp64 value and the
// fp64 remainder), so the reduced angle is accurate to ~1e-11 rad even at
// positions past 1e5.  GB300's fp64 rate is a small fraction of its fp32
// rate, so only the table kernel evaluates this; every other kernel reads
// the table.
constexpr double kTwoPiHi = 6.283185307179586;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189535;

// cos/sin of one angle as unevaluated fp32 pairs (hi + lo), from the fp64
// library sincos of the reduced angle: ~2^-48 accurate, enough to round a
// rotated key correctly even when x cos - y sin nearly cancels.
struct CosSin2 {
  float ch, cl, sh, sl;
};

__device__ __forceinline__ CosSin2 rope_cos_sin2(int pos, double inv_freq) {
  const double a = (double)pos * inv_freq;
  const double n = rint(a * kInvTwoPi);
  double r = fma(-n, kTwoPiHi, a);
  r = fma(-n, kTwoPiLo, r);
  double s, c;
  sincos(r, &s, &c);
  CosSin2 t;
  t.ch = (float)c;
  t.cl = (float)(c - (double)t.ch);
  t.sh = (float)s;
  t.sl = (float)(s - (double)t.sh);
  return t;
}

// a*(bh+bl) + c*(dh+dl) for fp32 a, c, as a double-float (hi, lo): exact
// products by FMA (TwoProduct) and exact TwoSums.  The _rn intrinsics keep
// the compiler from contracting the error-free steps into FMAs.
__device__ __forceinline__ void dot2_df(float a, float bh, float bl, float c, float dh, float dl, float& hi,
                                        float& lo) {
  const float p1 = __fmul_rn(a, bh);
  const float e1 = fmaf(a, bh, -p1);
  const float p2 = __fmul_rn(c, dh);
  const float e2 = fmaf(c, dh, -p2);
  const float s = __fadd_rn(p1, p2);
  const float bb = __fsub_rn(s, p1);
  const float es = __fadd_rn(__fsub_rn(p1, __fsub_rn(s, bb)), __fsub_rn(p2, bb));
  const float t = __fadd_rn(__fadd_rn(es, __fadd_rn(e1, e2)), fmaf(a, bl, __fmul_rn(c, dl)));
  hi = __fadd_rn(s, t);
  const float b2 = __fsub_rn(hi, s);
  lo = __fadd_rn(__fsub_rn(s, __fsub_rn(hi, b2)), __fsub_rn(t, b2));
}

// Rounds the double-float hi + lo to bf16 (nearest, ties to even).  Only an
// fp32 hi lying exactly on a bf16 midpoint needs lo to break the tie.
__device__ __forceinline__ uint32_t df_to_bf16_bits(float hi, float lo) {
  const uint32_t u = __float_as_uint(hi);
  const uint32_t low = u & 0xFFFFu;
  const uint32_t r = u >> 16;
  bool up;
  if (low != 0x8000u) up = low > 0x8000u;
  else if (lo == 0.f) up = (r & 1u) != 0;
  else up = (lo > 0.f) == (hi > 0.f);
  return r + (up ? 1u : 0u);
}

// a*(bh + bl) + c*(dh + dl) rounded once to bf16 (nearest even), for bf16-
// exact a, c and a double-float cos/sin (|bl| <= 2^-24 |bh|, same for d).
// Fast path: r = fma(a, bh, c*dh) in fp32 is within
// e = 2^-22 (|a bh| + |c dh|) of the exact value (the dropped lo terms, the
// product rounding and the fma rounding, each <= 2^-24 of those magnitudes);
// e is doubled against the rounding of the bound itself.  mid, the bf16
// midpoint inside r's bf16 interval, is the only midpoint within a quarter
// bf16 ulp (>= |r| 2^-10) of r, so with e below |r| 2^-10 and |r - mid|
// (exact) above e, r rounds like the exact value.  Otherwise (near a
// midpoint, or after heavy cancellation) the double-float evaluation, kept
// out of line, decides.
static __device__ __noinline__ uint32_t rot_bf16_bits_slow(float a, float bh, float bl, float c, float dh, float dl) {
  float hi, lo;
  dot2_df(a, bh, bl, c, dh, dl, hi, lo);
  return df_to_bf16_bits(hi, lo);
}

__device__ __forceinline__ uint32_t rot_bf16_bits(float a, float bh, float bl, float c, float dh, float dl) {
  const float p = __fmul_rn(c, dh);
  const float r = fmaf(a, bh, p);
  const float m = __fadd_rn(fabsf(__fmul_rn(a, bh)), fabsf(p));   // 2^21 e
  const uint32_t bits = __float_as_uint(r);
  const float mid = __uint_as_float((bits & 0xFFFF0000u) | 0x8000u);
  if (__fmul_rn(fabsf(__fsub_rn(r, mid)), 0x1p21f) > m && __fmul_rn(fabsf(r), 0x1p11f) > m)
    return (bits + 0x7FFFu + ((bits >> 16) & 1u)) >> 16;
  return rot_bf16_bits_slow(a, bh, bl, c, dh, dl);
}

// ---------------------------------------------------------------- bf16 helpers
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  f[0] = __uint_as_float(u.x << 16); f[1] = __uint_as_float(u.x & 0xffff0000u);
  f[2] = __uint_as_float(u.y << 16); f[3] = __uint_as_float(u.y & 0xffff0000u);
  f[4] = __uint_as_float(u.z << 16); f[5] = __uint_as_float(u.z & 0xffff0000u);
  f[6] = __uint_as_float(u.w << 16); f[7] = __uint_as_float(u.w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

// fp32 -> bf16 bits, round to nearest even (finite inputs)
__device__ __forceinline__ uint32_t bf16_bits_rn(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// 8 bf16 bit patterns (low 16 bits of each word) -> 16 bytes, element 0 first
__device__ __forceinline__ uint4 pack_bits8(const uint32_t (&h)[8]) {
  return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}

// Rotates 8 pairs: a holds elements [8c, 8c+8) of the first half, b the same
// offsets of the second half.  Each output is evaluated in double-float and
// rounded once to bf16, so it is the correctly rounded rotation of the
// stored bf16 inputs (to ~2^-44), also when x cos - y sin nearly cancels.
// t[e * STRIDE] holds the cos/sin of pair e of the 8 (a transposed shared-
// memory table uses STRIDE > 1 so that neighbouring lanes read neighbouring
// entries).
template <int STRIDE = 1>
__device__ __forceinline__ void rotate8_df(uint4& a, uint4& b, const CosSin2* t) {
  float x[8], y[8];
  unpack8(a, x);
  unpack8(b, y);
  uint32_t xo[8], yo[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const CosSin2 te = t[e * STRIDE];
    xo[e] = rot_bf16_bits(x[e], te.ch, te.cl, -y[e], te.sh, te.sl);   // x cos - y sin
    yo[e] = rot_bf16_bits(y[e], te.ch, te.cl, x[e], te.sh, te.sl);    // y cos + x sin
  }
  a = make_uint4(xo[0] | (xo[1] << 16), xo[2] | (xo[3] << 16), xo[4] | (xo[5] << 16), xo[6] | (xo[7] << 16));
  b = make_uint4(yo[0] | (yo[1] << 16), yo[2] | (yo[3] << 16), yo[4] | (yo[5] << 16), yo[6] | (yo[7] << 16));
}

// ---------------------------------------------------------------- mbarrier / bulk copy
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// 1-D bulk copy (TMA engine) global -> shared; bytes and both addresses must
// be multiples of 16.  Completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ---------------------------------------------------------------- kernel parameters

struct SegDesc {
  int32_t slot0;     // first composed row of this document
  int32_t n_slots;
  int32_t off;       // position offset: original tokens of the documents before it
  int32_t n_tokens;
};

// One document of a composition, in composed order.
struct ComposeSeg {
  const __nv_bfloat16* k;   // the document's pre-RoPE K [L][Hkv][n_slots][d] (pinned host pool, device address)
  const __nv_bfloat16* v;   // its V, same layout
  int32_t slot0;            // first composed row
  int32_t n_slots;
};

constexpr int kComposeCtas = 48;   // CTAs of one composition launch (~1.5 MB of host reads in flight)

struct ComposeParams {
  __nv_bfloat16* k_cache;   // [L][Hkv][cap][d]
  __nv_bfloat16* v_cache;
  const CosSin2* tab;       // [cap][d/2]: cos/sin of every cache row's position
  int32_t cap, n_kv, layer0, layer1, n_total, n_docs;
  ComposeSeg seg[kMaxDocsPerCompose];
};

// Builds the per-row cos/sin table (the only kernel that calls fp64 sincos).
struct TableParams {
  CosSin2* tab;              // [rows][d/2]
  int32_t* pos_out;          // optional [rows]
  const int32_t* pos_in;     // kTableExplicit: positions of the rows
  int32_t rows, half, mode;
  int32_t n_total, l_tot, k, n_docs;   // kTableComposed
  int32_t n_doc, kblk;                 // kTableExtraction
  double inv_freq[kMaxHalfDim];
  SegDesc seg[kMaxDocsPerCompose];
};

enum TableMode : int32_t { kTableComposed = 0, kTableExplicit = 1, kTableExtraction = 2 };

enum PosMode : int32_t { kPosSequential = 0, kPosExtraction = 1 };
enum MaskMode : int32_t { kMaskCausal = 0, kMaskStructured = 1, kMaskAnchor = 2 };

struct AppendParams {
  __nv_bfloat16* k_dst[kMaxBatch];   // layer base [Hkv][cap][d]
  __nv_bfloat16* v_dst[kMaxBatch];
  const CosSin2* tab[kMaxBatch];     // per-row cos/sin table of each sequence
  int32_t row_h[kMaxBatch];          // first destination row (host value) ...
  const int32_t* row_d;              // ... or device values (decode)
  const __nv_bfloat16* k_src;        // [B][t_len][Hkv][d]
  const __nv_bfloat16* v_src;
  const __nv_bfloat16* q_src;        // optional [B][t_len][Hq][d], rotated into ...
  __nv_bfloat16* q_dst;              // ... [B][Hkv][t_len][G][d] (bf16 hi part)
  __nv_bfloat16* q_dst_lo;           // and the same layout (bf16 lo part)
  unsigned* err;
  int32_t t_len, n_kv, n_q, cap;
};

// Tensor-core prefill: Q (hi and lo bf16 parts) from the rotated-q scratch
// [B][Hkv][t_len][G][d], K/V from 3-D maps {d, valid keys, layer * kv head}
// of each sequence's cache.
struct PrefillTcParams {
  const __nv_bfloat16* q_hi;
  const __nv_bfloat16* q_lo;
  CUtensorMap tm_k[kMaxBatch];
  CUtensorMap tm_v[kMaxBatch];
  int32_t n_cached[kMaxBatch];
  __nv_bfloat16* out;          // [B][t_len][Hq][d]
  unsigned* err;
  // num_splits key splits per unit, merged in a cluster of num_splits CTAs.
  // A unit is one (sequence, M tile, kv head), numbered (b * n_mt + mt) *
  // n_kv + h; a launch covers units [unit0, unit0 + n_units).
  int32_t batch, t_len, n_q, n_kv, layer, num_splits, split_keys, mask_mode, n_doc, kblk;
  int32_t n_mt, unit0, n_units;
  float scale_log2;
};

struct AttnParams {
  const __nv_bfloat16* k_base[kMaxBatch];   // layer base [Hkv][cap][d]
  const __nv_bfloat16* v_base[kMaxBatch];
  const CosSin2* tab[kMaxBatch];            // per-row cos/sin table: token t of
                                            // sequence b sits at row n_cached + t
  int32_t n_cached_h[kMaxBatch];
  const int32_t* n_cached_d;   // device lengths (decode) or null
  const __nv_bfloat16* q;      // [B][t_len][Hq][d]
  __nv_bfloat16* out;          // [B][t_len][Hq][d]
  float* part_o;               // [B][t_len][Hkv][S][G][d]
  float* part_ml;              // [B][t_len][Hkv][S][G][2]
  int32_t* counters;           // [B][token blocks][Hkv]
  unsigned* err;
  int32_t batch, t_len, n_q, n_kv, cap, max_keys;
  int32_t num_splits, split_keys;
  int32_t mask_mode, n_doc, kblk;
  // Decode with the append fused in: the new token's k (pre-RoPE) and v,
  // [B][Hkv][d]; the key is rotated, stored at row n_cached and used.
  int32_t fuse_append;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  // The num_splits CTAs of a (sequence, kv head) run as one thread-block
  // cluster and merge their partial results in distributed shared memory.
  int32_t cluster_merge;
  // Test hook (c2kv_test_expire_next_waits): the CTA's first tile wait also
  // waits on a barrier nothing arrives on, ~0.5 ms, and so takes the
  // timeout path.
  int32_t inject_timeout;
  float scale_log2;
};

// Decode on the tensor cores (head_dim 128): one launch per layer, the key
// tiles of all (sequence, kv head) units split evenly over one CTA per SM
// (decode_plan.h).  tm_k / tm_v: per sequence, a 3-D map {d, cap, kv heads}
// of this layer's cache, 64 x 128 x 1 boxes, 128-byte swizzle.
struct DecodeTcParams {
  CUtensorMap tm_k[kMaxBatch];
  CUtensorMap tm_v[kMaxBatch];
  __nv_bfloat16* k_base[kMaxBatch];   // layer base [Hkv][cap][d] (the fused append's rows)
  __nv_bfloat16* v_base[kMaxBatch];
  const CosSin2* tab[kMaxBatch];      // per-row cos/sin table of each sequence
  int32_t n_cached_h[kMaxBatch];      // host lengths (when n_cached_d is null)
  const int32_t* n_cached_d;          // device lengths
  const __nv_bfloat16* q;             // [B][Hq][d]
  __nv_bfloat16* out;                 // [B][Hq][d]
  const __nv_bfloat16* k_new;         // [B][Hkv][d] (fused append) or null
  const __nv_bfloat16* v_new;
  float* part_o;                      // [2 * CTAs][G][d] partial O of shared units
  float* part_ml;                     // [2 * CTAs][G][2] their (m, l)
  int32_t* counters;                  // [B * Hkv] tiles merged so far per unit
  unsigned* err;
  int32_t batch, n_q, n_kv, cap, max_keys;
  int32_t fuse_append, inject_timeout;
  // > 0: the launch is batch * n_kv thread-block clusters of `cluster` CTAs;
  // when every sequence has the same number of tiles (at least `cluster`),
  // cluster u holds exactly unit u and merges it in distributed shared memory
  int32_t cluster;
  float scale_log2;
};

// Linear layer on the tensor cores (linear_tc.cu): Y[t][n] = sum_k X[t][k] W[n][k]
// for t < tokens <= 256, with an epilogue.  tm_w: 2-D map {k_in, n_out} of W
// (box 64 x 128), tm_x: 2-D map {k_in, tokens} of X (box 64 x n_pad; rows past
// `tokens` read as zero), both with 128-byte swizzle.
enum LinearEpilogue : int32_t { kLinearStore = 0, kLinearAdd = 1, kLinearSplit3 = 2, kLinearSwiglu = 3 };
constexpr int kLinearSmemMax = 232448;
constexpr int kLinearSmemPerCta = 113 * 1024;   // two CTAs per SM (228 KB, 1 KB reserved per CTA)
struct LinearParams {
  CUtensorMap tm_w;
  CUtensorMap tm_x;
  const __nv_bfloat16* residual;   // kLinearAdd: [tokens][n_out] (may be y)
  __nv_bfloat16* y;                // [tokens][n_out]; kLinearSplit3: [tokens][split1];
  __nv_bfloat16* y2;               // kLinearSwiglu: [tokens][n_out / 2]
  __nv_bfloat16* y3;
  float* part;                     // [2 * CTAs][n_pad][128] partial tiles
  int32_t* counters;               // [n_out / 128] chunks summed so far per tile
  unsigned* err;
  int32_t tokens, n_pad, k_in, n_out, split1, split2, stages, epi;
  // 0: the (tile, chunk) items split evenly over the CTAs, partial tiles
  // merged through global memory by the last CTA of each tile.  cs >= 1: one
  // thread-block cluster of cs CTAs per tile, each CTA an equal share of the
  // tile's chunks, the cs partials summed through distributed shared memory
  // (cs = 1: every CTA one whole tile, nothing to merge).
  int32_t cs;
};

// Launchers (return cudaGetLastError()).
cudaError_t launch_linear(const LinearParams& p, int ctas, bool overlap, cudaStream_t st);
int linear_stages(int n_pad);
int linear_plan_cs(int n_out, int k_in, int n_pad, int ctas_max);   // LinearParams::cs
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* w, __nv_bfloat16* y, int tokens, int dim,
                           float eps, bool overlap, cudaStream_t st);
cudaError_t launch_decode_tc(const DecodeTcParams& p, int group, int ctas, bool overlap, cudaStream_t st);
// Clusters of `cs` CTAs of the tensor-core decode that fit the device at once
// (0 if unknown).
int decode_tc_active_clusters(int group, int cs);
cudaError_t launch_compose(const ComposeParams& p, int head_dim, cudaStream_t st);
cudaError_t launch_rope_table(const TableParams& p, cudaStream_t st);
cudaError_t launch_append(const AppendParams& p, int head_dim, int batch, cudaStream_t st);
cudaError_t launch_attention(const AttnParams& p, int head_dim, int group, bool overlap, cudaStream_t st);
cudaError_t launch_advance(int batch, int32_t* n_cached, int delta, cudaStream_t st);

cudaError_t launch_prefill_tc(const PrefillTcParams& p, int head_dim, int group, cudaStream_t st);
int prefill_tc_m_tiles(int t_len, int group);   // M tiles of 128 (token, head) rows
// Launches of one tensor-core prefill: units [0, bulk) in splits0 key splits
// of keys0 keys, then, if bulk < units, the rest in splits1 splits of keys1.
struct PrefillTcSchedule {
  int bulk, splits0, keys0, splits1, keys1;
};
PrefillTcSchedule prefill_tc_schedule(int units, int max_keys, int num_sms, int head_dim, int group, bool even);
int prefill_tc_key_tile();
// Key splits (one thread-block cluster per unit) and keys per split of the
// tensor-core prefill for `units` (sequence, M tile, kv head) units.
void prefill_tc_plan(int units, int max_keys, int num_sms, int head_dim, int group, int* num_splits,
                     int* split_keys);

// Attention work decomposition shared by the launcher and the workspace query.
int attn_tokens_per_cta(int t_len);
void attn_plan_splits(int units, int max_keys, int num_sms, int group, int* num_splits, int* split_keys);
int attn_cluster_splits(int units, int want, int head_dim, int group);

}  // namespace c2kv
