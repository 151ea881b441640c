// Split-K flash-decode over a composed cache, on CUDA cores.
//
// C2KV explainer (paper-daily.com), section "pipeline: extract, store,
// concatenate" (整体流程): after composition the question is appended and the
// answer generated over the concatenated cache; section "results"
// (实验结果：真的又快又准吗？): each decoded token reads the whole composed
// cache, so decode is bound by the bytes of that cache.  Section "structured
// information flow" (为什么需要“结构化信息流”？) gives the mask of the
// extraction-time mode (used here only for one-token sequences).
//
// One token per sequence.  A CTA owns one (sequence b, kv head h, key split)
// and is wide (16 warps, one wave of CTAs over the GPU) so that few splits
// cover a layer and their merge stays short.  The split's keys stream through
// a 3-stage ring of 128-key K/V tiles in shared memory, each tile fetched by
// two 1-D bulk copies (TMA engine) completing on an mbarrier; the first tiles
// are requested before anything else waits on memory.  The G q heads are
// split over warp slices of GW heads; a "key group" of d/16 lanes takes 4
// keys of every tile, lane li owning the 16-byte chunks li and li + d/16
// of each row (for d = 128 a RoPE pair), so partial dots use packed
// fma.rn.f32x2 and a transposed reduce-scatter over the group leaves one
// score per lane; scores are exchanged through shared memory.  Each group
// keeps its own online-softmax state (m, l, o), rescaled lazily (only when
// the running max grows by more than 2^8).  q is rotated once per CTA from
// the sequence's RoPE table and pre-scaled.  Groups are merged in shared
// memory; with several splits the CTA writes (m, l, o) partials, arrives on
// a per-(b, h) counter with one acq_rel atomic, and the last CTA to arrive
// merges them and resets the counter.  When a thread-block cluster of all
// the splits of every unit can be resident at once, the splits merge through
// distributed shared memory instead.
//
// Decode fuses the append: the CTA whose split holds the new key rotates it
// (correctly rounded to bf16, from the sequence's RoPE table), stores it with
// its value at row n_cached, and writes it into its last shared-memory tile,
// which the bulk copy leaves free; an mbarrier orders that write before the
// other warps read the tile.
#include <float.h>

#include <cooperative_groups.h>

#include "c2kv_internal.h"

namespace cg = cooperative_groups;

namespace c2kv {

namespace {

constexpr int kStages = 3;
constexpr int KPG = 4;   // keys per key group per tile

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
        "l"(*reinterpret_cast<unsigned long long*>(&c)));
  return *reinterpret_cast<float2*>(&r);
}

// 8 bf16 -> 4 fp32 pairs (element 2i in .x, 2i+1 in .y)
__device__ __forceinline__ void unpack8x2(const uint4& u, float2 (&f)[4]) {
  f[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
  f[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  f[2] = make_float2(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u));
  f[3] = make_float2(__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
}

template <int D, int G>
struct DCfg {
  // The G query heads of a kv head are split over HS warp slices of GW heads
  // each, so a thread holds q and o of GW heads only and 16 warps fit an SM.
  // An odd group (G = 5) would leave G one-head slices of 3 warps and
  // 48-key tiles; its warps take all G heads instead, 8 warps per CTA.
  static constexpr int GW = (G % 2 == 0) ? 2 : (G > 1 ? G : 1);   // heads per warp
  static constexpr int HS = G / GW;                   // head slices
  static constexpr int EPL = 16;                      // d elements a lane owns
  static constexpr int LPK = D / EPL;                 // lanes per key (a key group)
  static constexpr int NCH = EPL / 8;                 // 16-byte chunks a lane owns
  static constexpr int GPW = 32 / LPK;                // key groups per warp
  static constexpr int NWK0 = (GW > 2 ? 8 : 16) / HS;
  // warps per slice, halved while the 3-stage K/V ring would exceed 192 KB
  static constexpr int NWK1 = (NWK0 * GPW * KPG * D * 2 * 2 * kStages > 196608) ? NWK0 / 2 : NWK0;
  static constexpr int NWK = (NWK1 * GPW * KPG * D * 2 * 2 * kStages > 196608) ? NWK1 / 2 : NWK1;
  static constexpr int NW = HS * NWK;                 // warps per CTA
  static constexpr int THREADS = NW * 32;
  static constexpr int NG = NWK * GPW;                // key groups per slice
  static constexpr int T = NG * KPG;                  // keys per tile
  static constexpr int V = KPG * GW;                  // (key, head) scores a group makes per tile
  static constexpr int VP = ((V > LPK ? V : LPK) + LPK - 1) / LPK * LPK;   // padded to a multiple of LPK
  static constexpr int VPL = VP / LPK;                // scores each lane ends up owning
  static constexpr int TILE = T * D * 2;              // bytes of one K (or V) tile
  static constexpr int PIPE = kStages * 2 * TILE;
  static constexpr int CMB = NG * G * (D + 2) * 4;
  static constexpr int MAIN = ((PIPE > CMB ? PIPE : CMB) + 127) / 128 * 128;
  static constexpr int WN = NG > kMaxSplits ? NG : kMaxSplits;
  static constexpr int OFF_OCL = MAIN;                         // this split's O [G][D] for the cluster merge
  static constexpr int OFF_QS = OFF_OCL + G * D * 4;            // rotated, scaled q [G][D] fp32
  static constexpr int OFF_SC = OFF_QS + G * D * 4;             // per-group scores [HS][NG][VP]
  static constexpr int OFF_W = OFF_SC + HS * NG * VP * 4;       // merge weights [G][WN] + [G] M, L
  static constexpr int OFF_BAR = (OFF_W + G * WN * 4 + 2 * G * 4 + 15) / 16 * 16;
  static constexpr int OFF_CS = OFF_BAR + (2 * kStages + 3) * 8;   // merge flag
  static constexpr int SMEM = OFF_CS + 16;
  static_assert(G % GW == 0 && NWK >= 1 && NG % 2 == 0, "decode tiling");
};

// Sums VP partial values across the LPK lanes of a key group and scatters the
// totals: afterwards lane li holds, in x[0..VP/LPK), the totals of values
// [li * VP/LPK, (li+1) * VP/LPK).  Each step exchanges half of the current
// values with the partner lane (xor OFF), so VP - VP/LPK values cross lanes
// in all instead of VP * log2(LPK).
template <int N, int OFF, int VP>
struct ReduceScatter {
  __device__ __forceinline__ static void run(float (&x)[VP], int li) {
    if constexpr (OFF >= 1) {
      const bool up = (li & OFF) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = up ? x[i] : x[i + N / 2];
        const float keep = up ? x[i + N / 2] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
      }
      ReduceScatter<N / 2, OFF / 2, VP>::run(x, li);
    }
  }
};

// Extra visibility of the structured mask beyond causality (section
// "structured information flow"): slot i sees document tokens of the sink
// block [0, k) and of its own block [i*k, min((i+1)k, n_doc)) only.
__device__ __forceinline__ bool structured_visible(const AttnParams& p, int tok, int key) {
  if (tok < p.n_doc || key >= p.n_doc) return true;
  const int i = tok - p.n_doc;
  const int sink_end = min(p.kblk, p.n_doc);
  return key < sink_end || (key >= i * p.kblk && key < min((i + 1) * p.kblk, p.n_doc));
}

template <int D, int G>
__global__ void __launch_bounds__(DCfg<D, G>::THREADS, 1) decode_kernel(const __grid_constant__ AttnParams p) {
  using C = DCfg<D, G>;
  constexpr int T = C::T;
  constexpr int NW = C::NW;
  constexpr int LPK = C::LPK;
  constexpr int NCH = C::NCH;
  constexpr int TPR = D / 16;
  extern __shared__ __align__(1024) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem + C::OFF_QS);
  float* ocl = reinterpret_cast<float*>(smem + C::OFF_OCL);
  float* scs = reinterpret_cast<float*>(smem + C::OFF_SC);
  float* wbuf = reinterpret_cast<float*>(smem + C::OFF_W);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + kStages;
  uint64_t* inj = empty + kStages;                                     // new-key row injected
  uint64_t* never = inj + 1;                                           // test hook: nothing arrives
  int* flag = reinterpret_cast<int*>(smem + C::OFF_CS);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;

  const int n_cached = p.n_cached_d ? p.n_cached_d[b] : p.n_cached_h[b];
  if (n_cached < 0 || n_cached + 1 > p.cap || n_cached + 1 > p.max_keys) {
    // Uniform over every CTA of sequence b: nobody touches its counters.
    if (tid == 0 && split == 0 && h == 0) atomicOr(p.err, kErrLength);
    return;
  }
  const int kmax = n_cached + 1;   // the token sees every cached key and itself
  const int kb = split * p.split_keys;
  const int ke = min(kb + p.split_keys, kmax);
  const int ntiles = ke > kb ? (ke - kb + T - 1) / T : 0;
  const int nk = n_cached;         // index of the new key
  const bool has_new = p.fuse_append && nk >= kb && nk < ke;
  const int t_new = has_new ? (nk - kb) / T : -1;
  const int k_res_end = p.fuse_append ? min(ke, nk) : ke;   // end of cache-resident keys

  const __nv_bfloat16* kg = p.k_base[b] + (size_t)h * p.cap * D;
  const __nv_bfloat16* vg = p.v_base[b] + (size_t)h * p.cap * D;
  auto stage_k = [&](int s) { return smem + s * 2 * C::TILE; };
  auto stage_v = [&](int s) { return smem + s * 2 * C::TILE + C::TILE; };
  auto issue = [&](int t) {
    const int s = t % kStages;
    const int key0 = kb + t * T;
    const int cnt = max(0, min(T, k_res_end - key0));
    if (cnt == 0) {   // the tile holds only the new key
      mbar_arrive(&full[s]);
      return;
    }
    const uint32_t bytes = (uint32_t)cnt * D * 2;
    mbar_arrive_expect_tx(&full[s], 2 * bytes);
    bulk_g2s(stage_k(s), kg + (size_t)key0 * D, bytes, &full[s]);
    bulk_g2s(stage_v(s), vg + (size_t)key0 * D, bytes, &full[s]);
  };
  // The first tiles are requested before anything else waits on memory.
  int issued = 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    mbar_init(inj, TPR);
    mbar_init(never, 1);
    fence_barrier_init();
    for (; issued < min(kStages, ntiles); ++issued) issue(issued);
  }
  // Everything above reads only the lengths, the cache rows below n_cached
  // and nothing written since; with an overlapping launch (the caller's
  // C2KV_DECODE_OVERLAP_PREVIOUS) it runs while the previous kernel on the
  // stream finishes.  From here on the previous kernel must be complete:
  // q, the new k/v, the outputs and the scratch may be shared with it.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // q of the kv head's G query heads, rotated once per CTA (cos/sin from row
  // n_cached of the sequence's table) and pre-scaled by log2(e)/sqrt(d).
  const CosSin2* trow = p.tab[b] + (size_t)n_cached * (D / 2);
  for (int i = tid; i < G * (D / 2); i += C::THREADS) {
    const int g = i / (D / 2), f = i % (D / 2);
    const __nv_bfloat16* row = p.q + ((size_t)b * p.n_q + h * G + g) * D;
    const float x = __bfloat162float(row[f]), y = __bfloat162float(row[f + D / 2]);
    const float c = trow[f].ch, sn = trow[f].sh;
    qs[g * D + f] = (x * c - y * sn) * p.scale_log2;
    qs[g * D + f + D / 2] = (y * c + x * sn) * p.scale_log2;
  }
  __syncthreads();

  // ---- per-lane role: head slice hs (heads g0 .. g0+GW-1), key group gq;
  // lane li of the group owns the 16-byte chunks li, li + LPK of every row
  // (for d = 128 a RoPE pair; the 8 lanes of a group read 8 consecutive
  // chunks).
  constexpr int GW = C::GW;
  const int hs = warp / C::NWK;
  const int g0 = hs * GW;
  const int gq = (warp % C::NWK) * C::GPW + lane / LPK;
  const int li = lane % LPK;
  float2 q2[GW][NCH * 4];
#pragma unroll
  for (int g = 0; g < GW; ++g) {
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const float4* src = reinterpret_cast<const float4*>(qs + (g0 + g) * D + (li + j * LPK) * 8);
      const float4 a = src[0], c = src[1];
      q2[g][j * 4 + 0] = make_float2(a.x, a.y);
      q2[g][j * 4 + 1] = make_float2(a.z, a.w);
      q2[g][j * 4 + 2] = make_float2(c.x, c.y);
      q2[g][j * 4 + 3] = make_float2(c.z, c.w);
    }
  }

  float m[GW], l[GW];
  float2 o2[GW][NCH * 4];
#pragma unroll
  for (int g = 0; g < GW; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < NCH * 4; ++e) o2[g][e] = make_float2(0.f, 0.f);
  }

  // The new key's rotated k and v, prepared by warp 1 (lane c owns pairs
  // [8c, 8c+8)); written to the cache now and into the smem tile later.
  uint4 nk_a = make_uint4(0, 0, 0, 0), nk_b = nk_a, nv_a = nk_a, nv_b = nk_a;
  if (has_new && warp == 1 && lane < TPR) {
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_new + ((size_t)b * p.n_kv + h) * D);
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_new + ((size_t)b * p.n_kv + h) * D);
    nk_a = ks[lane];
    nk_b = ks[lane + TPR];
    nv_a = vs[lane];
    nv_b = vs[lane + TPR];
    rotate8_df(nk_a, nk_b, trow + lane * 8);
    uint4* kd = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(kg) + (size_t)nk * D);
    uint4* vd = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(vg) + (size_t)nk * D);
    kd[lane] = nk_a;
    kd[lane + TPR] = nk_b;
    vd[lane] = nv_a;
    vd[lane + TPR] = nv_b;
  }

  const bool structured = p.mask_mode == kMaskStructured;
  float* scg = scs + (hs * C::NG + gq) * C::VP;
  bool aborted = false;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % kStages;
    const uint32_t ph = (t / kStages) & 1;
    if (!mbar_wait(&full[s], ph)) { aborted = true; break; }
    if (p.inject_timeout && t == 0 && !mbar_wait(never, 0, kInjectWaitCycles)) { aborted = true; break; }
    if (t == t_new) {
      if (warp == 1 && lane < TPR) {
        const int r = nk - (kb + t * T);
        uint4* ksm = reinterpret_cast<uint4*>(stage_k(s) + (size_t)r * D * 2);
        uint4* vsm = reinterpret_cast<uint4*>(stage_v(s) + (size_t)r * D * 2);
        ksm[lane] = nk_a;
        ksm[lane + TPR] = nk_b;
        vsm[lane] = nv_a;
        vsm[lane + TPR] = nv_b;
        mbar_arrive(inj);
      }
      if (!mbar_wait(inj, 0)) { aborted = true; break; }
    }
    const int key0 = kb + t * T;
    const int nvalid = min(T, ke - key0);
    const uint8_t* Ks = stage_k(s);
    const uint8_t* Vs = stage_v(s);

    // partial q.k of this lane's chunks for the group's KPG keys x GW heads
    float x[C::VP];
#pragma unroll
    for (int kk = 0; kk < KPG; ++kk) {
      const int kl = kk * C::NG + gq;
      float2 k2[NCH * 4];
      if (kl < nvalid) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float2 t4[4];
          unpack8x2(*reinterpret_cast<const uint4*>(Ks + (size_t)kl * D * 2 + (li + j * LPK) * 16), t4);
#pragma unroll
          for (int e = 0; e < 4; ++e) k2[j * 4 + e] = t4[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < NCH * 4; ++e) k2[e] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int g = 0; g < GW; ++g) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < NCH * 4; ++e) a = ffma2(q2[g][e], k2[e], a);
        x[kk * GW + g] = a.x + a.y;
      }
    }
#pragma unroll
    for (int v = C::V; v < C::VP; ++v) x[v] = 0.f;
    ReduceScatter<C::VP, LPK / 2, C::VP>::run(x, li);
    // every lane of the group needs every score: exchange through shared memory
#pragma unroll
    for (int i = 0; i < C::VPL; ++i) scg[li * C::VPL + i] = x[i];
    __syncwarp();
    float sc[KPG][GW];
#pragma unroll
    for (int kk = 0; kk < KPG; ++kk) {
      const int kl = kk * C::NG + gq;
      bool vis = kl < nvalid;
      if (structured) vis = vis && structured_visible(p, n_cached, key0 + kl);
#pragma unroll
      for (int g = 0; g < GW; ++g) sc[kk][g] = vis ? scg[kk * GW + g] : -INFINITY;
    }
    __syncwarp();
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      float mc = sc[0][g];
#pragma unroll
      for (int kk = 1; kk < KPG; ++kk) mc = fmaxf(mc, sc[kk][g]);
      // Lazy rescale: keep the running max unless it grows by more than 2^8
      // (weights stay below 2^8; the final o / l is unaffected).
      if (mc > m[g] + 8.f || (m[g] == -INFINITY && mc > -INFINITY)) {
        const float a = exp2f(m[g] - mc);   // 0 when m was -inf
        l[g] *= a;
#pragma unroll
        for (int e = 0; e < NCH * 4; ++e) o2[g][e] = make_float2(o2[g][e].x * a, o2[g][e].y * a);
        m[g] = mc;
      }
    }
#pragma unroll
    for (int kk = 0; kk < KPG; ++kk) {
      const int kl = kk * C::NG + gq;
      if (kl < nvalid) {
        float2 v2[NCH * 4];
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          float2 t4[4];
          unpack8x2(*reinterpret_cast<const uint4*>(Vs + (size_t)kl * D * 2 + (li + j * LPK) * 16), t4);
#pragma unroll
          for (int e = 0; e < 4; ++e) v2[j * 4 + e] = t4[e];
        }
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          const float mu = (m[g] == -INFINITY) ? 0.f : m[g];
          const float pr = exp2f(sc[kk][g] - mu);
          l[g] += pr;
          const float2 p2 = make_float2(pr, pr);
#pragma unroll
          for (int e = 0; e < NCH * 4; ++e) o2[g][e] = ffma2(p2, v2[e], o2[g][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (tid == 0 && issued < ntiles) {
      if (!mbar_wait(&empty[s], ph)) { aborted = true; break; }
      issue(issued);
      ++issued;
    }
  }

  if (__syncthreads_or(aborted)) {
    // Let copies already in flight land before the shared memory is reused.
    if (tid == 0) {
      for (int t = max(0, issued - kStages); t < issued; ++t) mbar_wait(&full[t % kStages], (t / kStages) & 1);
      atomicOr(p.err, kErrTimeout);
    }
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < NCH * 4; ++e) o2[g][e] = make_float2(0.f, 0.f);
    }
    __syncthreads();
  }

  // ---- merge the key groups (pipeline shared memory reused)
  float* cmb_o = reinterpret_cast<float*>(smem);   // [NG][G][D]
  float* cmb_ml = cmb_o + C::NG * G * D;           // [NG][G][2]
#pragma unroll
  for (int gi = 0; gi < GW; ++gi) {
    const int g = g0 + gi;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      float4* dst = reinterpret_cast<float4*>(cmb_o + ((size_t)gq * G + g) * D + (li + j * LPK) * 8);
      dst[0] = make_float4(o2[gi][j * 4 + 0].x, o2[gi][j * 4 + 0].y, o2[gi][j * 4 + 1].x, o2[gi][j * 4 + 1].y);
      dst[1] = make_float4(o2[gi][j * 4 + 2].x, o2[gi][j * 4 + 2].y, o2[gi][j * 4 + 3].x, o2[gi][j * 4 + 3].y);
    }
    if (li == 0) {
      cmb_ml[(gq * G + g) * 2 + 0] = m[gi];
      cmb_ml[(gq * G + g) * 2 + 1] = l[gi];
    }
  }
  __syncthreads();
  // weight of group j for head g (one warp per head): w = 2^(m_j - M)
  float* wg = wbuf;                    // [G][NG]
  float* ML = wbuf + G * C::WN;        // [G][2]
  for (int g = warp; g < G; g += NW) {
    float M = -INFINITY;
    for (int j = lane; j < C::NG; j += 32) M = fmaxf(M, cmb_ml[(j * G + g) * 2]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int j = lane; j < C::NG; j += 32) {
      const float mj = cmb_ml[(j * G + g) * 2];
      const float w = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
      wg[g * C::WN + j] = w;
      L = fmaf(cmb_ml[(j * G + g) * 2 + 1], w, L);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) {
      ML[g * 2 + 0] = M;
      ML[g * 2 + 1] = L;
    }
  }
  __syncthreads();

  const int S = p.num_splits;
  for (int i = tid; i < G * D; i += C::THREADS) {
    const int dd = i % D, g = i / D;
    const float* w = wg + g * C::WN;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
    for (int j = 0; j < C::NG; j += 2) {
      a0 = fmaf(w[j], cmb_o[((size_t)j * G + g) * D + dd], a0);
      a1 = fmaf(w[j + 1], cmb_o[((size_t)(j + 1) * G + g) * D + dd], a1);
    }
    const float O = a0 + a1;
    if (p.cluster_merge) {
      ocl[g * D + dd] = O;
    } else if (S == 1) {
      p.out[((size_t)b * p.n_q + h * G + g) * D + dd] = __float2bfloat16_rn(O / ML[g * 2 + 1]);
    } else {
      const size_t base = ((size_t)b * p.n_kv + h) * S + split;
      p.part_o[(base * G + g) * D + dd] = O;
      if (dd == 0) {
        p.part_ml[(base * G + g) * 2 + 0] = ML[g * 2 + 0];
        p.part_ml[(base * G + g) * 2 + 1] = ML[g * 2 + 1];
      }
    }
  }
  if (p.cluster_merge) {
    // The splits of this (b, h) form one thread-block cluster: merge them
    // through distributed shared memory, each CTA producing every S-th output.
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();   // every split's O and (M, L) are in its shared memory
    const int r = (int)cl.block_rank();
    for (int i = r + S * tid; i < G * D; i += S * C::THREADS) {
      const int dd = i % D, g = i / D;
      float M = -INFINITY;
      for (int sp = 0; sp < S; ++sp) M = fmaxf(M, cl.map_shared_rank(ML, sp)[g * 2]);
      float L = 0.f, O = 0.f;
      for (int sp = 0; sp < S; ++sp) {
        const float* ml = cl.map_shared_rank(ML, sp);
        const float ms = ml[g * 2];
        const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
        L = fmaf(ml[g * 2 + 1], w, L);
        O = fmaf(cl.map_shared_rank(ocl, sp)[g * D + dd], w, O);
      }
      p.out[((size_t)b * p.n_q + h * G + g) * D + dd] = __float2bfloat16_rn(O / L);
    }
    cl.sync();   // no CTA leaves while others still read its shared memory
    return;
  }
  if (S == 1) return;

  // ---- last CTA of (b, h) merges the split partials.  The CTA barrier
  // orders every thread's partial stores before thread 0's acq_rel arrival
  // (release, cumulative); the last arriver's acquire, then the barrier,
  // orders its threads' partial loads after every split's stores.
  __syncthreads();
  const int cidx = b * p.n_kv + h;
  if (tid == 0) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(p.counters + cidx) : "memory");
    *flag = (prev == S - 1);
  }
  __syncthreads();
  if (!*flag) return;

  float* wts = wbuf;   // [G][S] (S <= WN)
  const size_t base = ((size_t)b * p.n_kv + h) * S;
  // The partial outputs of the first kPre splits of this thread's first
  // output are loaded now, in flight together with the (m, l) loads below.
  constexpr int kPre = 24;
  float pre[kPre];
  if (tid < G * D) {
    const float* po = p.part_o + (base * G + tid / D) * D + tid % D;
#pragma unroll
    for (int sp = 0; sp < kPre; ++sp) pre[sp] = sp < S ? __ldcg(po + (size_t)sp * G * D) : 0.f;
  }
  for (int g = warp; g < G; g += NW) {
    float M = -INFINITY;
    for (int sp = lane; sp < S; sp += 32) M = fmaxf(M, __ldcg(&p.part_ml[((base + sp) * G + g) * 2]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int sp = lane; sp < S; sp += 32) {
      const float ms = __ldcg(&p.part_ml[((base + sp) * G + g) * 2]);
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      wts[g * C::WN + sp] = w;
      L = fmaf(__ldcg(&p.part_ml[((base + sp) * G + g) * 2 + 1]), w, L);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float inv = 1.f / L;
    __syncwarp();
    for (int sp = lane; sp < S; sp += 32) wts[g * C::WN + sp] *= inv;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += C::THREADS) {
    const int dd = i % D, g = i / D;
    const float* w = wts + g * C::WN;
    const float* po = p.part_o + (base * G + g) * D + dd;
    // independent partial sums so the loads of several splits are in flight
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int sp = 0;
    if (i == tid) {
#pragma unroll
      for (int j = 0; j < kPre; j += 4) {
        a0 = fmaf(j + 0 < S ? w[j + 0] : 0.f, pre[j + 0], a0);
        a1 = fmaf(j + 1 < S ? w[j + 1] : 0.f, pre[j + 1], a1);
        a2 = fmaf(j + 2 < S ? w[j + 2] : 0.f, pre[j + 2], a2);
        a3 = fmaf(j + 3 < S ? w[j + 3] : 0.f, pre[j + 3], a3);
      }
      sp = kPre;
    }
    for (; sp + 4 <= S; sp += 4) {
      const float x0 = __ldcg(po + (size_t)(sp + 0) * G * D), x1 = __ldcg(po + (size_t)(sp + 1) * G * D);
      const float x2 = __ldcg(po + (size_t)(sp + 2) * G * D), x3 = __ldcg(po + (size_t)(sp + 3) * G * D);
      a0 = fmaf(w[sp + 0], x0, a0);
      a1 = fmaf(w[sp + 1], x1, a1);
      a2 = fmaf(w[sp + 2], x2, a2);
      a3 = fmaf(w[sp + 3], x3, a3);
    }
    for (; sp < S; ++sp) a0 = fmaf(w[sp], __ldcg(po + (size_t)sp * G * D), a0);
    p.out[((size_t)b * p.n_q + h * G + g) * D + dd] = __float2bfloat16_rn((a0 + a1) + (a2 + a3));
  }
  if (tid == 0) p.counters[cidx] = 0;
}

template <int D, int G>
KernelSetup& decode_setup() {
  static KernelSetup s;
  return s;
}

// Sets the kernel's attributes on device `dev` once (caller holds s.mu).
template <int D, int G>
cudaError_t configure_decode(KernelSetup& s, int dev) {
  using C = DCfg<D, G>;
  if (s.state[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(decode_kernel<D, G>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) cudaGetLastError();
    s.state[dev] = e == cudaSuccess ? 1 : -(int)e;
  }
  return s.state[dev] == 1 ? cudaSuccess : (cudaError_t)(-s.state[dev]);
}

template <int D, int G>
cudaError_t launch_one(const AttnParams& p, bool overlap, cudaStream_t st) {
  using C = DCfg<D, G>;
  {
    KernelSetup& s = decode_setup<D, G>();
    const int dev = setup_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(s.mu);
    const cudaError_t e = configure_decode<D, G>(s, dev);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits, p.n_kv, p.batch);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.cluster_merge) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p.num_splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, G>, p);
}

// Largest cluster of key splits (<= 16, one CTA per split) of which `units`
// clusters can be resident at once; 0 if none of size >= 2 fits.
template <int D, int G>
int cluster_splits_for(int units, int want) {
  using C = DCfg<D, G>;
  KernelSetup& s = decode_setup<D, G>();
  const int dev = setup_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lk(s.mu);
  if (configure_decode<D, G>(s, dev) != cudaSuccess) return 0;
  int* cache = s.clusters[dev];
  for (int cs = want < 16 ? want : 16; cs >= 2; --cs) {
    if (cache[cs] == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(C::THREADS);
      cfg.dynamicSmemBytes = C::SMEM;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<D, G>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = -1;
      }
      cache[cs] = n == 0 ? -1 : n;
    }
    if (cache[cs] >= units) return cs;
  }
  return 0;
}

template <int D>
int cluster_d(int units, int want, int group) {
  switch (group) {
    case 1: return cluster_splits_for<D, 1>(units, want);
    case 2: return cluster_splits_for<D, 2>(units, want);
    case 4: return cluster_splits_for<D, 4>(units, want);
    case 5: return cluster_splits_for<D, 5>(units, want);
    case 8: return cluster_splits_for<D, 8>(units, want);
    default: return 0;
  }
}

template <int D>
cudaError_t launch_d(const AttnParams& p, int group, bool overlap, cudaStream_t st) {
  switch (group) {
    case 1: return launch_one<D, 1>(p, overlap, st);
    case 2: return launch_one<D, 2>(p, overlap, st);
    case 4: return launch_one<D, 4>(p, overlap, st);
    case 5: return launch_one<D, 5>(p, overlap, st);
    case 8: return launch_one<D, 8>(p, overlap, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int attn_tokens_per_cta(int) { return 1; }

// One wave: units = sequences x kv heads; each unit's keys are split so that
// the CTAs (one wide CTA per SM) fill the SMs once.
void attn_plan_splits(int units, int max_keys, int num_sms, int group, int* num_splits, int* split_keys) {
  (void)group;
  int s = num_sms / units;
  if (s < 1) s = 1;
  if (s > kMaxSplits) s = kMaxSplits;
  const int min_keys = 64;   // keep each split at least a few tiles' worth of work
  if (s > 1 && (max_keys + s - 1) / s < min_keys) s = (max_keys + min_keys - 1) / min_keys;
  if (s < 1) s = 1;
  int sk = (max_keys + s - 1) / s;
  sk = (sk + 7) / 8 * 8;
  *split_keys = sk;
  *num_splits = (max_keys + sk - 1) / sk;
  if (*num_splits < 1) *num_splits = 1;
}

int attn_cluster_splits(int units, int want, int head_dim, int group) {
  if (want < 2) return 0;
  if (head_dim == 128) return cluster_d<128>(units, want, group);
  if (head_dim == 64) return cluster_d<64>(units, want, group);
  return 0;
}

cudaError_t launch_attention(const AttnParams& p, int head_dim, int group, bool overlap, cudaStream_t st) {
  if (p.t_len != 1) return cudaErrorInvalidValue;
  if (head_dim == 128) return launch_d<128>(p, group, overlap, st);
  if (head_dim == 64) return launch_d<64>(p, group, overlap, st);
  return cudaErrorInvalidValue;
}

}  // namespace c2kv
