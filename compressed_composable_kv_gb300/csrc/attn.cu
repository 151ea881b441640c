// Split-K flash attention over a composed cache, on CUDA cores.
//
// C2KV explainer (paper-daily.com), section "pipeline: extract, store,
// concatenate" (整体流程): after composition the question is appended and the
// answer generated over the concatenated cache; section "results"
// (实验结果：真的又快又准吗？): each decoded token reads the whole composed
// cache, so decode is bound by the bytes of that cache.  Section "structured
// information flow" (为什么需要“结构化信息流”？) gives the mask of the
// extraction-time mode.
//
// Work decomposition.  A CTA owns one (sequence b, kv head h, token block,
// key split).  Its key range is streamed through a 4-stage ring of 32-key
// K/V tiles in shared memory, each tile fetched by two 1-D bulk copies (TMA
// engine) completing on an mbarrier.  Rows are (token, q head of the group):
// the G heads of a token share every K/V tile.  A "key group" of D/8 lanes
// scores one key at a time (each lane holds 8 elements of d for all G heads,
// partial dots reduced with xor shuffles) and keeps its own online-softmax
// state (m, l, o); groups are merged through shared memory at the end.
// Decode (one token) spreads the 4 warps over the keys; prefill and the mask
// mode give each warp its own token.  With more than one split the CTA
// writes (m, l, o) partials; the last CTA of its (b, token block, h) to
// arrive (atomic counter) merges them and resets the counter.
#include <float.h>

#include "c2kv_internal.h"

namespace c2kv {

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kStages = 4;
constexpr int T = kAttnTileKeys;

template <int D, int G, int WPT>
struct Cfg {
  static constexpr int LPK = D / 8;          // lanes per key
  static constexpr int GPW = 32 / LPK;       // key groups per warp
  static constexpr int TPC = kWarps / WPT;   // tokens per CTA
  static constexpr int GPT = WPT * GPW;      // key groups per token
  static constexpr int KPG = T / GPT;        // keys per group per tile
  static constexpr int CH = KPG < 8 ? KPG : 8;
  static constexpr int TILE = T * D * 2;     // bytes of one K (or V) tile
  static constexpr int PIPE = kStages * 2 * TILE;
  static constexpr int CMB = TPC * GPT * G * (D + 2) * 4;
  static constexpr int WTS = TPC * G * kMaxSplits * 4;
  static constexpr int MAIN_RAW = (PIPE > CMB ? (PIPE > WTS ? PIPE : WTS) : (CMB > WTS ? CMB : WTS));
  static constexpr int MAIN = (MAIN_RAW + 127) / 128 * 128;   // keeps the mbarriers 8-byte aligned
  static constexpr int EXTRA = (2 * kStages + 2) * 8 + 2 * TPC * (D / 2) * 4 + (D / 2) * 16 + 16;
  static constexpr int SMEM = MAIN + EXTRA;
  static_assert(KPG >= 1 && KPG * GPT == T, "tile must split evenly over key groups");
};

// Extra visibility of the structured mask beyond causality (section
// "structured information flow"): slot i sees document tokens of the sink
// block [0, k) and of its own block [i*k, min((i+1)k, n_doc)) only.
// Document rows see no slot and slots see earlier slots; both follow from
// the causal limit because slots come after the document.
__device__ __forceinline__ bool structured_visible(const AttnParams& p, int tok, int key) {
  if (tok < p.n_doc || key >= p.n_doc) return true;
  const int i = tok - p.n_doc;
  const int sink_end = min(p.kblk, p.n_doc);
  return key < sink_end || (key >= i * p.kblk && key < min((i + 1) * p.kblk, p.n_doc));
}

template <int D, int G, int WPT>
__global__ void __launch_bounds__(kThreads) attn_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<D, G, WPT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::MAIN);
  uint64_t* empty = full + kStages;
  uint64_t* inj = empty + kStages;                          // new-key row injected (fused append)
  CosSin2* tab2 = reinterpret_cast<CosSin2*>(inj + 2);      // [D/2], position of the new key
  float* cs = reinterpret_cast<float*>(tab2 + D / 2);       // [TPC][D/2]
  float* sn = cs + C::TPC * (D / 2);
  int* flag = reinterpret_cast<int*>(sn + C::TPC * (D / 2));

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int h = blockIdx.y % p.n_kv;
  const int tb = blockIdx.y / p.n_kv;
  const int b = blockIdx.z;
  const int n_tb = (p.t_len + C::TPC - 1) / C::TPC;

  const int n_cached = p.n_cached_d ? p.n_cached_d[b] : p.n_cached_h[b];
  if (n_cached < 0 || n_cached + p.t_len > p.cap || n_cached + p.t_len > p.max_keys) {
    // Uniform over every CTA of sequence b: nobody touches its counters.
    if (tid == 0 && split == 0 && blockIdx.y == 0) atomicOr(p.err, kErrLength);
    return;
  }

  const int tok0 = tb * C::TPC;
  const int ntok = min(C::TPC, p.t_len - tok0);
  const int kmax = n_cached + tok0 + ntok;        // causal limit of the block's last token
  const int kb = split * p.split_keys;
  const int ke = min(kb + p.split_keys, kmax);
  const int ntiles = ke > kb ? (ke - kb + T - 1) / T : 0;
  // Fused append (decode): key nk = n_cached is the new token; the split that
  // holds it builds the row itself, every other key comes from the cache.
  constexpr int TPR = D / 16;
  const int nk = n_cached + p.t_len - 1;
  const bool has_new = p.fuse_append && nk >= kb && nk < ke;
  const int t_new = has_new ? (nk - kb) / T : -1;
  const int k_res_end = p.fuse_append ? min(ke, nk) : ke;   // end of cache-resident keys

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_init(inj, TPR);
    fence_barrier_init();
  }
  // cos/sin of each token's position: row n_cached + t of the sequence's table
  // (hi parts rotate q; the full pairs rotate the new key when fused).
  for (int i = tid; i < ntok * (D / 2); i += kThreads) {
    const int t = i / (D / 2), f = i % (D / 2);
    const CosSin2 e = p.tab[b][(size_t)(n_cached + tok0 + t) * (D / 2) + f];
    cs[i] = e.ch;
    sn[i] = e.sh;
    if (has_new && t == 0) tab2[f] = e;
  }
  __syncthreads();

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
  int issued = 0;
  if (tid == 0) {
    for (; issued < min(kStages, ntiles); ++issued) issue(issued);
  }

  // ---- per-lane role
  const int wtok = warp / WPT;
  const int gq = (warp % WPT) * C::GPW + lane / C::LPK;   // key group within token
  const int sub = lane % C::LPK;                          // owns d elements [8 sub, 8 sub + 8)
  const bool tok_ok = wtok < ntok;
  const int tok = tok0 + wtok;
  const int lim = n_cached + tok + 1;

  float q[G][8];
  {
    const int half = D / 2;
    const int e0 = sub * 8;
    const int partner = (e0 + half) % D;
    const float* c = cs + wtok * half;
    const float* s = sn + wtok * half;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x[8], y[8];
      if (tok_ok) {
        const __nv_bfloat16* row = p.q + (((size_t)b * p.t_len + tok) * p.n_q + h * G + g) * D;
        unpack8(*reinterpret_cast<const uint4*>(row + e0), x);
        unpack8(*reinterpret_cast<const uint4*>(row + partner), y);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = y[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int f = (e0 + e) % half;
        const float r = (e0 < half) ? x[e] * c[f] - y[e] * s[f] : x[e] * c[f] + y[e] * s[f];
        q[g][e] = r * p.scale_log2;
      }
    }
  }

  float m[G], l[G], o[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[g][e] = 0.f;
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
    rotate8_df(nk_a, nk_b, &tab2[lane * 8]);
    uint4* kd = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(kg) + (size_t)nk * D);
    uint4* vd = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(vg) + (size_t)nk * D);
    kd[lane] = nk_a;
    kd[lane + TPR] = nk_b;
    vd[lane] = nv_a;
    vd[lane + TPR] = nv_b;
  }

  bool aborted = false;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % kStages;
    const uint32_t ph = (t / kStages) & 1;
    if (!mbar_wait(&full[s], ph)) { aborted = true; break; }
    if (t == t_new) {
      // The row after the copied keys is free in this stage: fill it with the
      // new key, then let every warp read the tile.
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
#pragma unroll
    for (int c0 = 0; c0 < C::KPG; c0 += C::CH) {
      float sc[C::CH][G];
#pragma unroll
      for (int kk = 0; kk < C::CH; ++kk) {
        const int kl = (c0 + kk) * C::GPT + gq;
        const int key = key0 + kl;
        float kf[8];
        if (kl < nvalid) {
          unpack8(*reinterpret_cast<const uint4*>(Ks + (size_t)kl * D * 2 + sub * 16), kf);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) kf[e] = 0.f;
        }
        bool vis = tok_ok && kl < nvalid && key < lim;
        if (p.mask_mode == kMaskStructured) vis = vis && structured_visible(p, tok, key);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) d = fmaf(q[g][e], kf[e], d);
#pragma unroll
          for (int off = C::LPK / 2; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
          sc[kk][g] = vis ? d : -INFINITY;
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mc = sc[0][g];
#pragma unroll
        for (int kk = 1; kk < C::CH; ++kk) mc = fmaxf(mc, sc[kk][g]);
        if (mc > m[g]) {
          const float a = exp2f(m[g] - mc);   // 0 when m was -inf
          l[g] *= a;
#pragma unroll
          for (int e = 0; e < 8; ++e) o[g][e] *= a;
          m[g] = mc;
        }
      }
#pragma unroll
      for (int kk = 0; kk < C::CH; ++kk) {
        const int kl = (c0 + kk) * C::GPT + gq;
        if (kl < nvalid) {
          float vf[8];
          unpack8(*reinterpret_cast<const uint4*>(Vs + (size_t)kl * D * 2 + sub * 16), vf);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float mu = (m[g] == -INFINITY) ? 0.f : m[g];
            const float pr = exp2f(sc[kk][g] - mu);
            l[g] += pr;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[g][e] = fmaf(pr, vf[e], o[g][e]);
          }
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
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[g][e] = 0.f;
    }
    __syncthreads();
  }

  // ---- merge the key groups of each token (shared memory reused)
  float* cmb_o = reinterpret_cast<float*>(smem);              // [TPC][GPT][G][D]
  float* cmb_ml = cmb_o + C::TPC * C::GPT * G * D;             // [TPC][GPT][G][2]
  if (tok_ok) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* dst = cmb_o + (((size_t)wtok * C::GPT + gq) * G + g) * D + sub * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = o[g][e];
      if (sub == 0) {
        cmb_ml[((wtok * C::GPT + gq) * G + g) * 2 + 0] = m[g];
        cmb_ml[((wtok * C::GPT + gq) * G + g) * 2 + 1] = l[g];
      }
    }
  }
  __syncthreads();

  const int S = p.num_splits;
  for (int i = tid; i < ntok * G * D; i += kThreads) {
    const int dd = i % D, g = (i / D) % G, t = i / (G * D);
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < C::GPT; ++j) M = fmaxf(M, cmb_ml[((t * C::GPT + j) * G + g) * 2]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int j = 0; j < C::GPT; ++j) {
      const float mj = cmb_ml[((t * C::GPT + j) * G + g) * 2];
      const float w = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
      L = fmaf(cmb_ml[((t * C::GPT + j) * G + g) * 2 + 1], w, L);
      O = fmaf(cmb_o[((t * C::GPT + j) * G + g) * D + dd], w, O);
    }
    const int tk = tok0 + t;
    if (S == 1) {
      p.out[(((size_t)b * p.t_len + tk) * p.n_q + h * G + g) * D + dd] = __float2bfloat16_rn(O / L);
    } else {
      const size_t base = (((size_t)b * p.t_len + tk) * p.n_kv + h) * S + split;
      p.part_o[(base * G + g) * D + dd] = O;
      if (dd == 0) {
        p.part_ml[(base * G + g) * 2 + 0] = M;
        p.part_ml[(base * G + g) * 2 + 1] = L;
      }
    }
  }
  if (S == 1) return;

  // ---- last CTA of (b, token block, h) merges the split partials
  __threadfence();
  __syncthreads();
  const int cidx = (b * n_tb + tb) * p.n_kv + h;
  if (tid == 0) {
    const int prev = atomicAdd(&p.counters[cidx], 1);
    *flag = (prev == S - 1);
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();

  float* wts = reinterpret_cast<float*>(smem);   // [TPC][G][S]
  for (int pair = warp; pair < ntok * G; pair += kWarps) {
    const int t = pair / G, g = pair % G;
    const size_t base = (((size_t)b * p.t_len + tok0 + t) * p.n_kv + h) * S;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, __ldcg(&p.part_ml[((base + s) * G + g) * 2]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float ms = __ldcg(&p.part_ml[((base + s) * G + g) * 2]);
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      wts[pair * S + s] = w;
      L = fmaf(__ldcg(&p.part_ml[((base + s) * G + g) * 2 + 1]), w, L);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float invL = 1.f / L;
    __syncwarp();
    for (int s = lane; s < S; s += 32) wts[pair * S + s] *= invL;
  }
  __syncthreads();
  for (int i = tid; i < ntok * G * D; i += kThreads) {
    const int dd = i % D, g = (i / D) % G, t = i / (G * D);
    const size_t base = (((size_t)b * p.t_len + tok0 + t) * p.n_kv + h) * S;
    const float* w = wts + (t * G + g) * S;
    float acc = 0.f;
    for (int s = 0; s < S; ++s) acc = fmaf(w[s], __ldcg(&p.part_o[((base + s) * G + g) * D + dd]), acc);
    p.out[(((size_t)b * p.t_len + tok0 + t) * p.n_q + h * G + g) * D + dd] = __float2bfloat16_rn(acc);
  }
  if (tid == 0) p.counters[cidx] = 0;
}

template <int D, int G, int WPT>
cudaError_t launch_one(const AttnParams& p, cudaStream_t st) {
  using C = Cfg<D, G, WPT>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, G, WPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int n_tb = (p.t_len + C::TPC - 1) / C::TPC;
  const dim3 grid(p.num_splits, p.n_kv * n_tb, p.batch);
  attn_kernel<D, G, WPT><<<grid, kThreads, C::SMEM, st>>>(p);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_g(const AttnParams& p, cudaStream_t st) {
  // One token per sequence: the 4 warps split its keys.  Multi-token calls
  // go to the tensor-core kernel.
  if (p.t_len != 1) return cudaErrorInvalidValue;
  return launch_one<D, G, 4>(p, st);
}

template <int D>
cudaError_t launch_d(const AttnParams& p, int group, cudaStream_t st) {
  switch (group) {
    case 1: return launch_g<D, 1>(p, st);
    case 2: return launch_g<D, 2>(p, st);
    case 4: return launch_g<D, 4>(p, st);
    case 5: return launch_g<D, 5>(p, st);
    case 8: return launch_g<D, 8>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int attn_tokens_per_cta(int t_len) { return t_len == 1 ? 1 : kWarps; }


void attn_plan_splits(int units, int max_keys, int num_sms, int* num_splits, int* split_keys) {
  const int target = num_sms * kAttnCtasPerSm;
  int s = (target + units - 1) / units;
  const int tiles = (max_keys + T - 1) / T;
  if (s > tiles) s = tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s < 1) s = 1;
  int sk = (max_keys + s - 1) / s;
  sk = ((sk + T - 1) / T) * T;
  if (sk < T) sk = T;
  *split_keys = sk;
  *num_splits = (max_keys + sk - 1) / sk;
  if (*num_splits < 1) *num_splits = 1;
}

cudaError_t launch_attention(const AttnParams& p, int head_dim, int group, cudaStream_t st) {
  if (head_dim == 128) return launch_d<128>(p, group, st);
  if (head_dim == 64) return launch_d<64>(p, group, st);
  return cudaErrorInvalidValue;
}

}  // namespace c2kv
