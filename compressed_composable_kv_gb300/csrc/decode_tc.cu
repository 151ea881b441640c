// One decode step (one layer, a batch of sequences) on the 5th-generation
// tensor cores, head_dim 128.
//
// C2KV explainer (paper-daily.com), section "pipeline: extract, store,
// concatenate" (整体流程): after composition the question is appended and the
// answer generated over the concatenated cache; section "results"
// (实验结果：真的又快又准吗？): every generated token reads the whole composed
// cache, so decode is bound by the bytes of that cache, which C2KV shrinks.
//
// Work: the 128-key tiles of every (sequence b, kv head h) unit are laid end
// to end and cut into one equal contiguous range per CTA, one CTA per SM
// (decode_plan.h), from the device-side lengths; sequences of any lengths
// keep every SM streaming.  A CTA walks its range as segments (the part of
// one unit it owns).  A segment that covers a whole unit writes the output;
// otherwise the CTA writes a partial (m, l, O) and adds its tile count to the
// unit's counter, and the CTA whose addition completes the count merges.
//
// Per tile, with keys as the MMA's M dimension and the G query heads of the
// kv head as N (q split into bf16 hi + lo halves, 2G <= 16 columns, so the
// product keeps fp32-level accuracy):
//   K, V : 128 keys x 128 d, TMA (3-D map, 128-byte swizzle), 3-stage ring
//   S^T  = K q^T        tcgen05.mma M=128 N=16 K=128 -> TMEM (2 buffers)
//   softmax: thread t owns key t (TMEM lane t): s = S_hi + S_lo (q carries
//         log2(e)/sqrt(d)), tile max per head across the 4 warps, a running
//         reference max per head kept unless a tile's max exceeds it by 2^8,
//         p = 2^(s - m), written as bf16 hi + lo rows of P^T
//   O^T  = V^T P^T      tcgen05.mma M=128 (d) N=16 K=128 (keys), V read
//         MN-major from the same tile -> TMEM (2 buffers)
//   thread t (now d = t) accumulates o[g] = o[g] * alpha + O_hi + O_lo in
//         registers; each thread sums its keys' p into l.
// Roles: warps 0-3 softmax and epilogue, warp 4 lane 0 TMA, warp 5 lane 0
// MMA, warp 6 the rotated q of each segment and the new key.
//
// The append is fused: the CTA owning a unit's last tile rotates the new key
// (correctly rounded, from the sequence's RoPE table), stores it with its
// value at row n_cached, and writes both into the landed tile; rows past the
// valid keys of that tile are zeroed in V (they may hold any bits) and
// masked in the softmax.
#include <float.h>

#include <cooperative_groups.h>

#include "c2kv_internal.h"
#include "decode_plan.h"
#include "tcgen05.h"

namespace cg = cooperative_groups;

namespace c2kv {

namespace {

constexpr int DT_D = 128;
constexpr int DT_BN = kDecKeyTile;       // keys per tile
constexpr int DT_STAGES = 3;
constexpr int DT_THREADS = 224;
constexpr int DT_SM_THREADS = 128;       // softmax / epilogue threads (warps 0-3)
constexpr float kDtRescaleLog2 = 8.f;
constexpr int kMergeChunk = 8;           // partials whose loads are in flight together

struct DtCfg {
  static constexpr int KV_SUB = DT_BN * 128;              // [128 keys][64 d] bf16, one swizzle column block
  static constexpr int KV_BYTES = 2 * KV_SUB;             // K (or V) of one stage
  static constexpr int STAGE = 2 * KV_BYTES;              // K + V
  static constexpr int N_SUB = 16 * 128;                  // [16 rows][64] bf16
  static constexpr int QP_BYTES = 2 * N_SUB;              // one q (or P^T) operand [16 rows][128]
  static constexpr int OFF_KV = 0;
  static constexpr int OFF_Q = OFF_KV + DT_STAGES * STAGE;
  static constexpr int OFF_P = OFF_Q + 2 * QP_BYTES;
  static constexpr int OFF_RED = OFF_P + 2 * QP_BYTES;    // [2][4 warps][8] per-warp maxima / sums
  static constexpr int OFF_MAP = OFF_RED + 2 * 4 * 8 * 4;
  static constexpr int OFF_NC = OFF_MAP + (int)((sizeof(DecodeMap) + 15) / 16 * 16);   // [16] lengths
  static constexpr int OFF_SLOTS = OFF_NC + kDecMaxSeqs * 4;       // merge: slot of each contributor
  static constexpr int OFF_STML = OFF_SLOTS + kDecMaxCtas * 4;      // cluster merge: staged m [8], l [8]
  static constexpr int OFF_BAR = OFF_STML + 16 * 4;
  static constexpr int N_BAR = 2 * DT_STAGES + 2 * 8 + 5;
  static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;   // + slack for 1024-byte alignment
  static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzled operands need 1024-byte alignment");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static constexpr int TMEM_S = 0;      // two 16-column S^T buffers
  static constexpr int TMEM_O = 32;     // two 16-column O^T buffers
  static constexpr int TMEM_COLS = 64;
};

constexpr uint32_t kIdescQK = idesc_bf16_m128(16, false, false);   // A = K (K-major), B = q (K-major)
constexpr uint32_t kIdescPV = idesc_bf16_m128(16, true, false);    // A = V^T (MN-major), B = P^T (K-major)

// Columns of the TMEM loads: the G hi columns and the G lo columns.
template <int G>
struct DtCols {
  static constexpr int NC = 2 * G <= 2 ? 2 : 2 * G <= 4 ? 4 : 2 * G <= 8 ? 8 : 16;
};

// One segment: the tiles [j0, j0 + n) of the CTA's range, all of unit (b, h),
// starting at tile t0 of the unit.
struct DtSeg {
  int b, h, t0, j0, n;
};

__device__ __forceinline__ DtSeg seg_at(const DecodeMap& m, int64_t x0, int64_t x1, int j) {
  const DecodeTile d = decode_locate(m, x0 + j);
  DtSeg s;
  s.b = d.b;
  s.h = d.h;
  s.t0 = d.t;
  s.j0 = j;
  s.n = (int)min((int64_t)(m.tb[d.b] - d.t), x1 - (x0 + j));
  return s;
}

template <int G>
__global__ void __launch_bounds__(DT_THREADS, 1) decode_tc_kernel(const __grid_constant__ DecodeTcParams p) {
  using C = DtCfg;
  constexpr int NC = DtCols<G>::NC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = kv_full + DT_STAGES;
  uint64_t* s_full = kv_empty + DT_STAGES;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* p_free = p_full + 2;
  uint64_t* o_full = p_free + 2;
  uint64_t* o_free = o_full + 2;
  uint64_t* q_full = o_free + 2;
  uint64_t* q_free = q_full + 2;
  // A unit's last tile: the MMA thread signals fix_req once it has landed,
  // warp 6 writes the new key and zeroes the tail, then arrives on fix_bar.
  uint64_t* fix_req = q_free + 2;
  uint64_t* fix_bar = fix_req + 1;
  uint64_t* grp_bar = fix_bar + 1;    // the softmax warps' group barrier
  uint64_t* mma_done = grp_bar + 1;   // every MMA of the CTA has completed
  uint64_t* never = mma_done + 1;     // test hook: nothing arrives
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  volatile int* aligned_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 24);
  float* stml = reinterpret_cast<float*>(smem + C::OFF_STML);
  DecodeMap& M = *reinterpret_cast<DecodeMap*>(smem + C::OFF_MAP);
  int32_t* ncs = reinterpret_cast<int32_t*>(smem + C::OFF_NC);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);   // [2][4][8]
  int32_t* mslots = reinterpret_cast<int32_t*>(smem + C::OFF_SLOTS);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;

  if (tid == 0) {
    // Lengths: read before waiting for the previous kernel (they are not
    // among what it may write).  A bad length skips its sequence.
    int32_t keys[kDecMaxSeqs];
    bool bad = false;
    for (int b = 0; b < kDecMaxSeqs; ++b) {
      int32_t n = -1;
      if (b < p.batch) {
        n = p.n_cached_d ? p.n_cached_d[b] : p.n_cached_h[b];
        if (n < 0 || n + 1 > p.cap || n + 1 > p.max_keys) {
          bad = true;
          n = -1;
        }
      }
      ncs[b] = n;
      keys[b] = n + 1;
    }
    if (bad && cta == 0) atomicOr(p.err, kErrLength);
    decode_map_build(M, keys, p.batch, p.n_kv, (int)gridDim.x);
    // One cluster per unit (the cluster merge) when every sequence has the
    // same number of tiles, at least one per CTA of the cluster.
    bool al = p.cluster > 0 && !bad && M.tb[0] >= p.cluster &&
              (int)gridDim.x == p.batch * p.n_kv * p.cluster;
    for (int b = 1; b < p.batch; ++b) al = al && M.tb[b] == M.tb[0];
    *aligned_flag = al ? 1 : 0;
    for (int g = 0; g < 8; ++g) {
      stml[g] = -INFINITY;   // staged (m, l) of a CTA that never finishes its segment
      stml[8 + g] = 0.f;
    }
    for (int s = 0; s < DT_STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], DT_SM_THREADS);
      mbar_init(&p_full[i], DT_SM_THREADS);
      mbar_init(&p_free[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], DT_SM_THREADS);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_free[i], 1);
    }
    mbar_init(fix_req, 1);
    mbar_init(fix_bar, 1);
    mbar_init(grp_bar, 4);
    mbar_init(mma_done, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  uint8_t* sKV = smem + C::OFF_KV;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sP = smem + C::OFF_P;
  auto stage_k = [&](int s) { return sKV + s * C::STAGE; };
  auto stage_v = [&](int s) { return sKV + s * C::STAGE + C::KV_BYTES; };
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr((const void*)tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 6) {
    // rows 2G..15 of the q and P^T operands are never written: keep them zero
    for (int i = lane; i < 4 * C::QP_BYTES / 16; i += 32)
      reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t x0 = decode_cta_first(M, cta), x1 = decode_cta_first(M, cta + 1);
  const int ntiles = (int)(x1 - x0);
  if (ntiles == 0) {   // uniform over the CTA (never in a cluster-merged launch)
    if (warp == 4)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
    return;
  }
  const bool aligned = *aligned_flag != 0;
  int issued = 0;   // the TMA thread's count of tiles requested

  if (warp == 4) {
    if (lane == 0) {
      // ---------------- TMA producer: cache rows only, so it does not wait for
      // the previous kernel (rows at or past n_cached are fixed up in shared
      // memory before use).
      DecodeTile d = decode_locate(M, x0);
      for (int j = 0; j < ntiles; ++j, d = decode_next(M, d)) {
        const int s = j % DT_STAGES;
        if (j >= DT_STAGES && !wait_or_abort(&kv_empty[s], ((j - DT_STAGES) / DT_STAGES) & 1, abort_flag, p.err))
          break;
        mbar_arrive_expect_tx(&kv_full[s], C::STAGE);
        for (int sub = 0; sub < 2; ++sub) {
          tma_load_3d(stage_k(s) + sub * C::KV_SUB, &p.tm_k[d.b], sub * 64, d.t * DT_BN, d.h, &kv_full[s]);
          tma_load_3d(stage_v(s) + sub * C::KV_SUB, &p.tm_v[d.b], sub * 64, d.t * DT_BN, d.h, &kv_full[s]);
        }
        ++issued;
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------- MMA issuer
      auto issue_pv = [&](int i) -> bool {
        const int pb = i & 1, s = i % DT_STAGES;
        if (!wait_or_abort(&p_full[pb], (i >> 1) & 1, abort_flag, p.err)) return false;
        if (i >= 2 && !wait_or_abort(&o_free[pb], ((i - 2) >> 1) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DT_BN / 16; ++kk) {
          const uint64_t a = sw128_desc(smem_addr(stage_v(s)) + kk * 2048, C::KV_SUB, 1024);
          const uint64_t b = sw128_desc(smem_addr(sP + pb * C::QP_BYTES + (kk / 4) * C::N_SUB) + (kk % 4) * 32, 16, 1024);
          mma_bf16(tmem + C::TMEM_O + pb * 16, a, b, kIdescPV, kk > 0 ? 1u : 0u);
        }
        mma_commit(&kv_empty[s]);
        mma_commit(&p_free[pb]);
        mma_commit(&o_full[pb]);
        return true;
      };
      bool ok = true;
      int seg = -1, fixes = 0;
      DecodeTile d = decode_locate(M, x0);
      for (int j = 0; ok && j < ntiles; ++j, d = decode_next(M, d)) {
        const bool first = j == 0 || d.t == 0;
        const bool unit_last = d.t == M.tb[d.b] - 1;
        const bool seg_last = j == ntiles - 1 || unit_last;
        if (first) ++seg;
        const int s = j % DT_STAGES;
        ok = wait_or_abort(&kv_full[s], (j / DT_STAGES) & 1, abort_flag, p.err);
        if (ok && first) ok = wait_or_abort(&q_full[seg & 1], (seg >> 1) & 1, abort_flag, p.err);
        if (ok && unit_last) {
          mbar_arrive(fix_req);
          ok = wait_or_abort(fix_bar, (fixes++) & 1, abort_flag, p.err);
        }
        if (ok && j >= 2) ok = wait_or_abort(&s_free[j & 1], ((j - 2) >> 1) & 1, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DT_D / 16; ++kk) {
          const int sub = kk / 4, ko = (kk % 4) * 32;
          const uint64_t a = sw128_desc(smem_addr(stage_k(s) + sub * C::KV_SUB) + ko, 16, 1024);
          const uint64_t b = sw128_desc(smem_addr(sQ + (seg & 1) * C::QP_BYTES + sub * C::N_SUB) + ko, 16, 1024);
          mma_bf16(tmem + C::TMEM_S + (j & 1) * 16, a, b, kIdescQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[j & 1]);
        if (seg_last) mma_commit(&q_free[seg & 1]);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(ntiles - 1);
      // every MMA issued above must complete before TMEM is released
      mma_commit(mma_done);
      mbar_wait(mma_done, 0);
    }
  } else if (warp == 6) {
    // ---------------- rotated q of each segment, the new key of each unit the
    // CTA finishes
    // The first segment's cos/sin (the table is not written by the previous
    // kernel) are loaded before waiting for it; q and the new key after.
    constexpr int kItems = (G * 8 + 31) / 32;   // 8-pair items of q per lane
    DtSeg cur = seg_at(M, x0, x1, 0);
    float2 cs0[kItems][8];
    {
      const CosSin2* trow = p.tab[cur.b] + (size_t)ncs[cur.b] * (DT_D / 2);
#pragma unroll
      for (int it = 0; it < kItems; ++it) {
        const int item = lane + 32 * it;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const CosSin2 t = item < G * 8 ? trow[(item & 7) * 8 + e] : CosSin2{0.f, 0.f, 0.f, 0.f};
          cs0[it][e] = make_float2(t.ch, t.sh);
        }
      }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    auto prep_q = [&](int i, const DtSeg& sg) -> bool {
      if (i >= 2 && !__all_sync(0xffffffffu, wait_or_abort(&q_free[i & 1], ((i - 2) >> 1) & 1, abort_flag, p.err)))
        return false;
      const int n = ncs[sg.b];
      const CosSin2* trow = p.tab[sg.b] + (size_t)n * (DT_D / 2);
      uint8_t* qb = sQ + (i & 1) * C::QP_BYTES;
#pragma unroll
      for (int it = 0; it < kItems; ++it) {
        const int item = lane + 32 * it;
        if (item >= G * 8) break;
        const int g = item >> 3, c = item & 7;   // pairs f = 8c .. 8c+7 of head g
        const uint4* row = reinterpret_cast<const uint4*>(p.q + ((size_t)sg.b * p.n_q + sg.h * G + g) * DT_D);
        float x[8], y[8];
        unpack8(row[c], x);
        unpack8(row[c + 8], y);
        float h0[8], l0[8], h1[8], l1[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float2 t;
          if (i == 0) {
            t = cs0[it][e];
          } else {
            const CosSin2 tt = trow[c * 8 + e];
            t = make_float2(tt.ch, tt.sh);
          }
          const float a = (x[e] * t.x - y[e] * t.y) * p.scale_log2;
          const float b = (y[e] * t.x + x[e] * t.y) * p.scale_log2;
          h0[e] = __bfloat162float(__float2bfloat16_rn(a));
          l0[e] = a - h0[e];
          h1[e] = __bfloat162float(__float2bfloat16_rn(b));
          l1[e] = b - h1[e];
        }
        const int rh = g, rl = G + g;
        *reinterpret_cast<uint4*>(qb + rh * 128 + ((c ^ (rh & 7)) << 4)) = pack8(h0);
        *reinterpret_cast<uint4*>(qb + rl * 128 + ((c ^ (rl & 7)) << 4)) = pack8(l0);
        *reinterpret_cast<uint4*>(qb + C::N_SUB + rh * 128 + ((c ^ (rh & 7)) << 4)) = pack8(h1);
        *reinterpret_cast<uint4*>(qb + C::N_SUB + rl * 128 + ((c ^ (rl & 7)) << 4)) = pack8(l1);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full[i & 1]);
      return true;
    };
    // The last tile of unit (b, h), CTA tile j: new key in (fused append),
    // V rows past the valid keys zeroed.  The fixups come in tile order, as
    // the MMA thread's requests do.
    int fixes = 0;
    auto fixup = [&](int j, const DtSeg& sg) -> bool {
      const int n = ncs[sg.b];
      const int key0 = (sg.t0 + (j - sg.j0)) * DT_BN;
      const int r = n - key0;   // row of the new key in the tile (0..127)
      uint4 nk_a = make_uint4(0, 0, 0, 0), nk_b = nk_a, nv_a = nk_a, nv_b = nk_a;
      if (p.fuse_append && lane < 8) {
        const uint4* ks = reinterpret_cast<const uint4*>(p.k_new + ((size_t)sg.b * p.n_kv + sg.h) * DT_D);
        const uint4* vs = reinterpret_cast<const uint4*>(p.v_new + ((size_t)sg.b * p.n_kv + sg.h) * DT_D);
        nk_a = ks[lane];
        nk_b = ks[lane + 8];
        nv_a = vs[lane];
        nv_b = vs[lane + 8];
        rotate8_df(nk_a, nk_b, p.tab[sg.b] + (size_t)n * (DT_D / 2) + lane * 8);
        uint4* kd = reinterpret_cast<uint4*>(p.k_base[sg.b] + ((size_t)sg.h * p.cap + n) * DT_D);
        uint4* vd = reinterpret_cast<uint4*>(p.v_base[sg.b] + ((size_t)sg.h * p.cap + n) * DT_D);
        kd[lane] = nk_a;
        kd[lane + 8] = nk_b;
        vd[lane] = nv_a;
        vd[lane + 8] = nv_b;
      }
      // The request comes once the tile has landed, so the stage's current
      // fill is this tile's and its wait below returns at once.
      const int s = j % DT_STAGES;
      if (!__all_sync(0xffffffffu, wait_or_abort(fix_req, (fixes++) & 1, abort_flag, p.err))) return false;
      if (!__all_sync(0xffffffffu, wait_or_abort(&kv_full[s], (j / DT_STAGES) & 1, abort_flag, p.err))) return false;
      if (p.fuse_append && lane < 8) {
        const int sw = (lane ^ (r & 7)) << 4;
        *reinterpret_cast<uint4*>(stage_k(s) + r * 128 + sw) = nk_a;
        *reinterpret_cast<uint4*>(stage_k(s) + C::KV_SUB + r * 128 + sw) = nk_b;
        *reinterpret_cast<uint4*>(stage_v(s) + r * 128 + sw) = nv_a;
        *reinterpret_cast<uint4*>(stage_v(s) + C::KV_SUB + r * 128 + sw) = nv_b;
      }
      for (int i = lane; i < (DT_BN - 1 - r) * 16; i += 32) {
        const int row = r + 1 + (i >> 4), ch = i & 15;
        *reinterpret_cast<uint4*>(stage_v(s) + (ch >> 3) * C::KV_SUB + row * 128 + ((ch & 7) << 4)) =
            make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(fix_bar);
      return true;
    };
    bool ok = prep_q(0, cur);
    for (int i = 0; ok; ++i) {
      const bool more = cur.j0 + cur.n < ntiles;
      DtSeg nxt = cur;
      if (more) {
        nxt = seg_at(M, x0, x1, cur.j0 + cur.n);
        ok = prep_q(i + 1, nxt);
      }
      if (ok && cur.t0 + cur.n == M.tb[cur.b]) ok = fixup(cur.j0 + cur.n - 1, cur);
      if (!more) break;
      cur = nxt;
    }
  } else {
    // ---------------- softmax and epilogue: thread tid owns key tid of each
    // tile (TMEM lane tid of S^T) and output element d = tid (lane of O^T)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    int k_sync = 0;
    bool ok = true;
    int arrived = -1;   // last segment whose tiles were added to its unit's counter
    int i = 0;
    DtSeg sg = seg_at(M, x0, x1, 0);
    for (;; ++i) {
      const int n = ncs[sg.b];
      const int nkeys = n + 1;
      const bool whole = sg.t0 == 0 && sg.n == M.tb[sg.b];
      float m_ref[G], l_part[G], o_acc[G], a_prev[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m_ref[g] = -INFINITY;
        l_part[g] = 0.f;
        o_acc[g] = 0.f;
        a_prev[g] = 0.f;
      }
      auto consume_o = [&](int jj, const float (&alpha)[G]) -> bool {
        if (!__all_sync(0xffffffffu, wait_or_abort(&o_full[jj & 1], (jj >> 1) & 1, abort_flag, p.err))) return false;
        tc_fence_after();
        float ov[NC];
        tmem_ld_cols<NC>(lane_base + C::TMEM_O + (jj & 1) * 16, ov);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&o_free[jj & 1]);
#pragma unroll
        for (int g = 0; g < G; ++g) o_acc[g] = fmaf(o_acc[g], alpha[g], ov[g] + ov[G + g]);
        return true;
      };
      for (int tt = 0; ok && tt < sg.n; ++tt) {
        const int j = sg.j0 + tt;
        const int sb = j & 1;
        const int key0 = (sg.t0 + tt) * DT_BN;
        if (p.inject_timeout && j == 0 &&
            !__all_sync(0xffffffffu, mbar_wait(never, 0, kInjectWaitCycles))) {
          *abort_flag = 1;
          atomicOr(p.err, kErrTimeout);
          ok = false;
          break;
        }
        if (!__all_sync(0xffffffffu, wait_or_abort(&s_full[sb], (j >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[NC];
        tmem_ld_cols<NC>(lane_base + C::TMEM_S + sb * 16, sv);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
        const bool valid = key0 + tid < nkeys;
        float s[G];
        float* rb = red + (k_sync & 1) * 32;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          s[g] = valid ? sv[g] + sv[G + g] : -INFINITY;
          const float wm = warp_max(s[g]);
          if (lane == 0) rb[warp * 8 + g] = wm;
        }
        if (!group_sync(grp_bar, k_sync, abort_flag, p.err)) {
          ok = false;
          break;
        }
        float alpha[G];
        __nv_bfloat16 ph[G], pl[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float tmax = fmaxf(fmaxf(rb[g], rb[8 + g]), fmaxf(rb[16 + g], rb[24 + g]));
          alpha[g] = 1.f;
          if (m_ref[g] == -INFINITY) {
            alpha[g] = 0.f;   // nothing accumulated yet
            m_ref[g] = tmax;
          } else if (tmax > m_ref[g] + kDtRescaleLog2) {
            alpha[g] = exp2f(m_ref[g] - tmax);
            m_ref[g] = tmax;
          }
          const float pr = ex2_approx(s[g] - m_ref[g]);   // masked keys: 2^-inf = 0
          l_part[g] = fmaf(l_part[g], alpha[g], pr);
          ph[g] = __float2bfloat16_rn(pr);
          pl[g] = __float2bfloat16_rn(pr - __bfloat162float(ph[g]));
        }
        if (j >= 2 && !__all_sync(0xffffffffu, wait_or_abort(&p_free[sb], ((j - 2) >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        {
          uint8_t* pb = sP + sb * C::QP_BYTES + (tid >> 6) * C::N_SUB;
          const int e = tid & 63;
          const int off = (e & 7) * 2;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const int rh = g, rl = G + g;
            *reinterpret_cast<__nv_bfloat16*>(pb + rh * 128 + (((e >> 3) ^ (rh & 7)) << 4) + off) = ph[g];
            *reinterpret_cast<__nv_bfloat16*>(pb + rl * 128 + (((e >> 3) ^ (rl & 7)) << 4) + off) = pl[g];
          }
        }
        fence_proxy_async();
        mbar_arrive(&p_full[sb]);
        if (tt > 0 && !consume_o(j - 1, a_prev)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) a_prev[g] = alpha[g];
      }
      if (ok) ok = consume_o(sg.j0 + sg.n - 1, a_prev);

      // ---------------- segment epilogue
      const int u = sg.b * p.n_kv + sg.h;
      float L[G];
      if (ok) {
        float* rb = red + (k_sync & 1) * 32;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float ls = warp_sum(l_part[g]);
          if (lane == 0) rb[warp * 8 + g] = ls;
        }
        ok = group_sync(grp_bar, k_sync, abort_flag, p.err);
#pragma unroll
        for (int g = 0; g < G; ++g) L[g] = (rb[g] + rb[8 + g]) + (rb[16 + g] + rb[24 + g]);
      }
      if (ok && whole) {
#pragma unroll
        for (int g = 0; g < G; ++g)
          p.out[((size_t)sg.b * p.n_q + sg.h * G + g) * DT_D + tid] = __float2bfloat16_rn(o_acc[g] / L[g]);
      } else if (ok && aligned) {
        // the cluster merges the unit after the teardown: stage this CTA's
        // partial in shared memory (the P^T buffers are free: every PV has
        // completed)
        float* st_o = reinterpret_cast<float*>(sP);   // [G][d]
#pragma unroll
        for (int g = 0; g < G; ++g) {
          st_o[g * DT_D + tid] = o_acc[g];
          if (tid == g) {
            stml[g] = m_ref[g];
            stml[8 + g] = L[g];
          }
        }
      } else if (ok) {
        const int slot = 2 * cta + (i == 0 ? 0 : 1);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          p.part_o[((size_t)slot * G + g) * DT_D + tid] = o_acc[g];
          if (tid == g) {
            p.part_ml[((size_t)slot * G + g) * 2 + 0] = m_ref[g];
            p.part_ml[((size_t)slot * G + g) * 2 + 1] = L[g];
          }
        }
        // every partial store of the CTA is ordered before tid 0's arrival
        // (a release at GPU scope, cumulative over the group barrier)
        ok = group_sync(grp_bar, k_sync, abort_flag, p.err);
        if (ok && tid == 0) {
          int prev;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                       : "=r"(prev)
                       : "l"(p.counters + u), "r"(sg.n)
                       : "memory");
          const bool last = prev + sg.n == M.tb[sg.b];
          if (last) p.counters[u] = 0;   // every CTA of the unit has arrived
          *last_flag = last ? 1 : 0;
          arrived = i;
        }
        if (ok) ok = group_sync(grp_bar, k_sync, abort_flag, p.err);
        if (ok && *last_flag) {
          // ---- merge the unit's partials (the last CTA to arrive): the
          // contributors' slots go to shared memory once, then the partials
          // are read kMergeChunk at a time with every load in flight and
          // combined with a running max.
          const int64_t uf = M.start[sg.b] + (int64_t)sg.h * M.tb[sg.b];
          const int cf = decode_cta_of(M, uf), cl = decode_cta_of(M, uf + M.tb[sg.b] - 1);
          const int nctr = cl - cf + 1;
          for (int k = tid; k < nctr; k += DT_SM_THREADS)
            mslots[k] = decode_cta_empty(M, cf + k) ? -1 : decode_slot_of(M, cf + k, uf);
          ok = group_sync(grp_bar, k_sync, abort_flag, p.err);
          float mx[G], lt[G], ot[G];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            mx[g] = -INFINITY;
            lt[g] = 0.f;
            ot[g] = 0.f;
          }
          for (int k0 = 0; ok && k0 < nctr; k0 += kMergeChunk) {
            float mv[kMergeChunk][G], lv[kMergeChunk][G], ov[kMergeChunk][G];
#pragma unroll
            for (int k = 0; k < kMergeChunk; ++k) {
              const int sl = k0 + k < nctr ? mslots[k0 + k] : -1;
#pragma unroll
              for (int g = 0; g < G; ++g) {
                const size_t r = (size_t)(sl < 0 ? 0 : sl) * G + g;
                mv[k][g] = sl < 0 ? -INFINITY : __ldcg(&p.part_ml[r * 2]);
                lv[k][g] = sl < 0 ? 0.f : __ldcg(&p.part_ml[r * 2 + 1]);
                ov[k][g] = sl < 0 ? 0.f : __ldcg(&p.part_o[r * DT_D + tid]);
              }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float cm = mx[g];
#pragma unroll
              for (int k = 0; k < kMergeChunk; ++k) cm = fmaxf(cm, mv[k][g]);
              if (cm == -INFINITY) continue;
              const float sc = mx[g] == -INFINITY ? 0.f : exp2f(mx[g] - cm);
              lt[g] *= sc;
              ot[g] *= sc;
#pragma unroll
              for (int k = 0; k < kMergeChunk; ++k) {
                const float w = mv[k][g] == -INFINITY ? 0.f : exp2f(mv[k][g] - cm);
                lt[g] = fmaf(w, lv[k][g], lt[g]);
                ot[g] = fmaf(w, ov[k][g], ot[g]);
              }
              mx[g] = cm;
            }
          }
          if (ok) {
#pragma unroll
            for (int g = 0; g < G; ++g)
              p.out[((size_t)sg.b * p.n_q + sg.h * G + g) * DT_D + tid] = __float2bfloat16_rn(ot[g] / lt[g]);
          }
        }
      }
      if (!ok) break;
      if (sg.j0 + sg.n >= ntiles) break;
      sg = seg_at(M, x0, x1, sg.j0 + sg.n);
    }
    if (!ok && tid == 0 && !aligned) {
      // The CTA gave up: still add the tiles of its remaining shared units to
      // their counters (their outputs are undefined), so every counter is back
      // at zero when the launch ends.  (A cluster-merged launch uses none.)
      DtSeg q = seg_at(M, x0, x1, 0);
      for (int k = 0;; ++k) {
        const bool whole_q = q.t0 == 0 && q.n == M.tb[q.b];
        if (k > arrived && !whole_q) {
          const int u = q.b * p.n_kv + q.h;
          const int prev = atomicAdd(p.counters + u, q.n);
          if (prev + q.n == M.tb[q.b]) p.counters[u] = 0;
        }
        if (q.j0 + q.n >= ntiles) break;
        q = seg_at(M, x0, x1, q.j0 + q.n);
      }
    }
  }

  // ---------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 4 && lane == 0) {
    // let the copies in flight land before the shared memory is released
    for (int j = max(0, issued - DT_STAGES); j < issued; ++j) mbar_wait(&kv_full[j % DT_STAGES], (j / DT_STAGES) & 1);
  }
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
  }
  if (aligned) {
    // ---------------- cluster merge: the cluster is the unit's CTAs; CTA r
    // writes its share of the G x d outputs from every CTA's staged partial.
    // Every CTA reaches both cluster barriers on every path (all waits above
    // are bounded; a CTA that gave up stages m = -inf and adds nothing), and
    // none leaves before its peers' reads of its shared memory are done.
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();
    const int CS = p.cluster;
    const int r = (int)cl.block_rank();
    const int unit = cta / CS;
    const int b = unit / p.n_kv, h = unit % p.n_kv;
    const int per = (G * DT_D + CS - 1) / CS;
    const float* st_o = reinterpret_cast<const float*>(sP);
    for (int e = r * per + tid; e < min(G * DT_D, (r + 1) * per); e += DT_THREADS) {
      const int g = e / DT_D, d = e % DT_D;
      float mx = -INFINITY;
      for (int sp = 0; sp < CS; ++sp) mx = fmaxf(mx, cl.map_shared_rank(stml, sp)[g]);
      float lt = 0.f, ot = 0.f;
      for (int sp = 0; sp < CS; ++sp) {
        const float ms = cl.map_shared_rank(stml, sp)[g];
        const float w = ms == -INFINITY ? 0.f : exp2f(ms - mx);
        lt = fmaf(w, cl.map_shared_rank(stml, sp)[8 + g], lt);
        ot = fmaf(w, cl.map_shared_rank(st_o, sp)[g * DT_D + d], ot);
      }
      p.out[((size_t)b * p.n_q + h * G + g) * DT_D + d] = __float2bfloat16_rn(ot / lt);
    }
    cl.sync();
  }
}

template <int G>
KernelSetup& dtc_setup() {
  static KernelSetup s;
  return s;
}

// Sets the kernel's attributes on device `dev` once (caller holds s.mu).
template <int G>
cudaError_t configure_dtc(KernelSetup& s, int dev) {
  if (s.state[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, DtCfg::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_tc_kernel<G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) cudaGetLastError();
    s.state[dev] = e == cudaSuccess ? 1 : -(int)e;
  }
  return s.state[dev] == 1 ? cudaSuccess : (cudaError_t)(-s.state[dev]);
}

template <int G>
cudaError_t launch_dtc(const DecodeTcParams& p, int ctas, bool overlap, cudaStream_t st) {
  {
    KernelSetup& s = dtc_setup<G>();
    const int dev = setup_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(s.mu);
    const cudaError_t e = configure_dtc<G>(s, dev);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(DT_THREADS);
  cfg.dynamicSmemBytes = DtCfg::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.cluster > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p.cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<G>, p);
}

template <int G>
int dtc_active_clusters(int cs) {
  if (cs < 2 || cs > 16) return 0;
  KernelSetup& s = dtc_setup<G>();
  const int dev = setup_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lk(s.mu);
  if (configure_dtc<G>(s, dev) != cudaSuccess) return 0;
  int* cache = s.clusters[dev];
  if (cache[cs] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(DT_THREADS);
    cfg.dynamicSmemBytes = DtCfg::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<G>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[cs] = n > 0 ? n : -1;
  }
  return cache[cs] > 0 ? cache[cs] : 0;
}

}  // namespace

int decode_tc_active_clusters(int group, int cs) {
  switch (group) {
    case 1: return dtc_active_clusters<1>(cs);
    case 2: return dtc_active_clusters<2>(cs);
    case 4: return dtc_active_clusters<4>(cs);
    case 5: return dtc_active_clusters<5>(cs);
    case 8: return dtc_active_clusters<8>(cs);
    default: return 0;
  }
}

cudaError_t launch_decode_tc(const DecodeTcParams& p, int group, int ctas, bool overlap, cudaStream_t st) {
  switch (group) {
    case 1: return launch_dtc<1>(p, ctas, overlap, st);
    case 2: return launch_dtc<2>(p, ctas, overlap, st);
    case 4: return launch_dtc<4>(p, ctas, overlap, st);
    case 5: return launch_dtc<5>(p, ctas, overlap, st);
    case 8: return launch_dtc<8>(p, ctas, overlap, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace c2kv
