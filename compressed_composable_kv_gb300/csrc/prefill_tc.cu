// Question prefill (and the extraction mask mode) on the 5th-generation
// tensor cores: QK^T and PV run as tcgen05.mma with TMEM accumulators.
//
// C2KV explainer (paper-daily.com), section "pipeline: extract, store,
// concatenate" (整体流程): once the composed cache is in place the question is
// appended and prefilled over it; section "structured information flow"
// (为什么需要“结构化信息流”？) gives the extraction-time mask; section
// "results" gives the anchor-token ablation's mask.
//
// One CTA owns a 128-row M tile of (question token, q head of the group)
// rows for one (sequence, kv head, key split), token-major and packed across
// tokens: row r of tile mt is token (128 mt + r) / G, head (128 mt + r) % G.
// Warps 0-3 are the softmax warps (thread t owns row t, i.e. TMEM lane t);
// one lane of warp 4 issues the QK MMAs and one of warp 7 the PV MMAs, so
// neither kind waits behind the other's issue; warps 5 and 6 issue the K and
// the V loads.  Everything the tensor
// cores read besides K and V sits in TMEM, so shared memory holds only the
// two load rings.
//   Q   : [128 rows][d] as bf16 hi + lo parts (hi + lo within ~2^-16 of the
//         rotated q), loaded by the softmax threads (thread = row) into TMEM;
//         S = Q_hi K^T + Q_lo K^T takes A from TMEM, so the logits keep
//         fp32-level accuracy (a bf16 q alone errs by ~2^-9 of |q||k|, which a
//         sharp softmax turns into output errors near the tolerance)
//   K,V : 128-key tiles, TMA (3-D map over [layer*kv head][keys][d]), a ring
//         of 3 stages each (a tile load takes ~2 us from L2, so 2 stages left
//         the tensor pipe waiting); keys at or past the sequence's valid
//         length read as zeros (OOB); key tiles no row of the M tile can see
//         are skipped
//   S   : Q K^T, fp32 in TMEM, two buffers of 128 columns: QK(j + 1) runs
//         while the softmax works on S(j)
//   P   : bf16 in TMEM over the first 64 columns of its own S buffer (two
//         keys per column); PV takes A = P from TMEM.  QK(j + 2), the next
//         write of that buffer, is issued after PV(j), and tcgen05.mma
//         operations of one thread run in issue order
//   O   : P V accumulated in TMEM (d columns), rescaled in place only when a
//         row's running max grows by more than 2^8 (the final O / l uses the
//         same stale max, so the result is exact)
// With several key splits, the S split CTAs of one (sequence, M tile, kv
// head) form a thread-block cluster: each stages its unnormalised O (fp32)
// and (m, l) in shared memory, and after a cluster barrier CTA r merges rows
// [r * ceil(128 / S), ...) of all S splits through distributed shared memory
// and writes them, so no partial result goes through global memory.
#include <cuda.h>

#include <algorithm>

#include <cooperative_groups.h>

#include "c2kv_internal.h"
#include "tcgen05.h"

namespace cg = cooperative_groups;

namespace c2kv {

namespace {

constexpr int BM = 128;        // rows per M tile (TMEM lanes)
constexpr int BN = 128;        // keys per tile
constexpr int STAGES = 3;      // K ring and V ring depth (each its own barriers)
constexpr int kMaxClusterTc = 16;   // key splits merged in one cluster
constexpr int kSoftmaxThreads = 128;
constexpr int kThreadsTc = 256;   // warps 0-3 softmax, 4 QK MMAs, 5 K loads, 6 V loads, 7 PV MMAs
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct TcCfg {
  static constexpr int NSUB = D / 64;           // 128-byte column blocks of d
  static constexpr int KV_BYTES = NSUB * BN * 128;
  static constexpr int MRG_BYTES = (BM + kMaxClusterTc) * 3 * 4;   // split merge: m, l, weights
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  // split merge (after the last PV, when the V ring is free): (m, l) of
  // every row and the merge's m, l and weights, over the V ring
  static constexpr int OFF_ML = OFF_V;
  static constexpr int OFF_MRG = OFF_ML + BM * 2 * 4;
  static_assert(OFF_MRG + MRG_BYTES <= OFF_V + STAGES * KV_BYTES, "merge scratch must fit the V ring");
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr int N_BAR = 1 + 4 * STAGES + 2 + 2 + 2 + 1;   // q, K/V rings, S, P, PV, last PV
  static constexpr int OFF_MISC = OFF_BAR + N_BAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;   // + slack for 1024-byte alignment
  // split merge: unnormalised O of every row (fp32, 16-byte chunks swizzled
  // by row & 7) over the K ring, merge weights over the Q tile
  static constexpr int OFF_OST = OFF_K;
  static_assert(BM * D * 4 <= STAGES * KV_BYTES, "O staging must fit the K ring");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  // S: two buffers of BN columns; P(j) (bf16, two keys per column) is
  // written over the first BN / 2 columns of S(j)'s buffer once S(j) is read
  static constexpr int TMEM_S = 0;
  static constexpr int TMEM_O = 2 * BN;               // d columns
  static constexpr int TMEM_QH = 3 * BN;              // Q_hi: d / 2 columns (two bf16 per column)
  static constexpr int TMEM_QL = TMEM_QH + D / 2;     // Q_lo
  static constexpr int TMEM_COLS = 512;
  static_assert(TMEM_O + D <= TMEM_QH && TMEM_QL + D / 2 <= TMEM_COLS, "TMEM columns");
};

__device__ __forceinline__ bool tc_structured_visible(const PrefillTcParams& p, int tok, int key) {
  if (tok < p.n_doc || key >= p.n_doc) return true;
  const int i = tok - p.n_doc;
  return key < min(p.kblk, p.n_doc) || (key >= i * p.kblk && key < min((i + 1) * p.kblk, p.n_doc));
}

// MASKED: the extraction masks (structured, anchor); the question prefill
// runs the causal instantiation, which carries no mask code.
template <int D, int G, bool MASKED>
__global__ void __launch_bounds__(kThreadsTc, 1) prefill_tc_kernel(const __grid_constant__ PrefillTcParams p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  // K and V stages are filled and freed separately: a K stage is free once
  // its QK^T has run, a V stage once its PV has.
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + STAGES;
  uint64_t* v_full = k_empty + STAGES;
  uint64_t* v_empty = v_full + STAGES;
  uint64_t* s_full = v_empty + STAGES;
  uint64_t* p_full = s_full + 2;
  // PV(t) completes phase t >> 1 of o_done[t & 1], so a wait for PV(j-1)
  // can never mistake an older phase of the same parity for it; o_last
  // (single use) completes with the last PV of the CTA.
  uint64_t* o_done = p_full + 2;
  uint64_t* o_last = o_done + 2;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  volatile int* k_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 24);   // K loads issued
  volatile int* v_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 28);   // V loads issued

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // the num_splits CTAs of a unit are consecutive in x and form its cluster
  const int split = (int)blockIdx.x % p.num_splits;
  const int unit = p.unit0 + (int)blockIdx.x / p.num_splits;
  const int h = unit % p.n_kv;
  const int mt = unit / p.n_kv % p.n_mt;
  const int b = unit / (p.n_kv * p.n_mt);
  const int n_cached = p.n_cached[b];
  // The (token, head) rows of the question are packed 128 to an M tile,
  // token-major: tile mt holds rows [128 mt, 128 mt + 128) of the t_len * G,
  // so a token's heads may straddle two tiles (G = 5: 5 tiles for 128 tokens
  // instead of 6 of 25 tokens each).
  const int r_tile = mt * BM;
  const int n_rows = p.t_len * G;
  const int tok0 = r_tile / G;                                  // first token with a row here
  const int ntok = min((r_tile + BM - 1) / G + 1, p.t_len) - tok0;
  // Anchor-token mask: document rows also see every anchor, so an M tile
  // holding document rows reads the keys of the whole sequence.
  const int mode = MASKED ? p.mask_mode : (int)kMaskCausal;
  const bool anchor_docs = mode == kMaskAnchor && tok0 < p.n_doc;
  const int kmax = n_cached + (anchor_docs ? p.t_len : tok0 + ntok);
  const int kb = split * p.split_keys;
  const int ke = min(kb + p.split_keys, kmax);
  const int ntiles = ke > kb ? (ke - kb + BN - 1) / BN : 0;
  // Structured mask ("structured information flow"): an M tile of slot rows
  // only sees the sink block, its own slots' document blocks and the slots,
  // so the other document key tiles hold no visible key and are skipped.
  // Anchor mask: document key tiles past the M tile's last row hold no key
  // its rows see (they see the anchors and their causal prefix).  The masked
  // modes run with no cached rows, so key index = token index.
  // Every role walks the same list of live tiles.
  auto tile_live = [&](int t) -> bool {
    if (anchor_docs) {
      const int key0 = kb + t * BN;
      return key0 < tok0 + ntok || key0 + BN > p.n_doc;
    }
    if (mode != kMaskStructured || tok0 < p.n_doc) return true;   // document rows: causal
    const int key0 = kb + t * BN;
    if (key0 + BN > p.n_doc || key0 < min(p.kblk, p.n_doc)) return true;  // slot keys, sink block
    const int lo = (tok0 - p.n_doc) * p.kblk;
    const int hi = min((tok0 + ntok - p.n_doc) * p.kblk, p.n_doc);
    return key0 < hi && key0 + BN > lo;
  };
  auto next_live = [&](int t) -> int {
    while (t < ntiles && !tile_live(t)) ++t;
    return t;
  };
  int nlive = 0;
  for (int t = 0; t < ntiles; ++t) nlive += tile_live(t) ? 1 : 0;

  if (tid == 0) {
    mbar_init(q_full, kSoftmaxThreads);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxThreads);
    }
    mbar_init(&o_done[0], 1);
    mbar_init(&o_done[1], 1);
    mbar_init(o_last, 1);
    *abort_flag = 0;
    *k_issued = 0;
    *v_issued = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr((const void*)tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The launch of the rest of the last wave (prefill_tc_schedule) reads
  // nothing this one writes: its CTAs may take the SMs this launch frees.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  const int kv_z = p.layer * p.n_kv + h;

  float m_run = -INFINITY, l_run = 0.f;   // softmax threads: running max / sum of their row
  if (warp == 5 || warp == 6) {
    if (lane == 0 && nlive > 0) {
      // ---------------- producers: warp 5 loads the live K tiles, warp 6 the
      // V tiles; the jj-th live tile goes to stage jj % STAGES of its ring
      const bool is_k = warp == 5;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = is_k ? sK : sV;
      const CUtensorMap* map = is_k ? &p.tm_k[b] : &p.tm_v[b];
      volatile int* issued = is_k ? k_issued : v_issued;
      int t = next_live(0);
      for (int jj = 0; jj < nlive; ++jj, t = next_live(t + 1)) {
        const int s = jj % STAGES;
        if (jj >= STAGES && !wait_or_abort(&empty[s], ((jj - STAGES) / STAGES) & 1, abort_flag, p.err)) break;
        mbar_arrive_expect_tx(&full[s], C::KV_BYTES);
        for (int sub = 0; sub < C::NSUB; ++sub)
          tma_load_3d(ring + s * C::KV_BYTES + sub * BN * 128, map, sub * 64, kb + t * BN, kv_z, &full[s]);
        *issued = jj + 1;
      }
    }
  } else if (warp == 4) {
    if (lane == 0 && nlive > 0) {
      // ---------------- QK issuer (one thread): QK(j) into S buffer j & 1
      // once PV(j - 2), which read P(j - 2) from that buffer, has completed
      constexpr uint32_t IDESC_QK = idesc_bf16_m128(BN, false, false);
      auto issue_qk = [&](int j) -> bool {
        const int s = j % STAGES;
        if (!wait_or_abort(&k_full[s], (j / STAGES) & 1, abort_flag, p.err)) return false;
        if (j >= 2 && !wait_or_abort(&o_done[j & 1], ((j - 2) >> 1) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t d = tmem + C::TMEM_S + (j & 1) * BN;
#pragma unroll
        for (int half = 0; half < 2; ++half) {   // Q_hi K^T, then + Q_lo K^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int sub = kk / 4, ko = (kk % 4) * 32;
            const uint64_t bdesc = sw128_desc(smem_addr(sK + s * C::KV_BYTES + sub * BN * 128) + ko, 16, 1024);
            mma_bf16_tmem_a(d, tmem + (half ? C::TMEM_QL : C::TMEM_QH) + kk * 8, bdesc, IDESC_QK,
                            (half | kk) ? 1u : 0u);
          }
        }
        mma_commit(&k_empty[s]);
        mma_commit(&s_full[j & 1]);
        return true;
      };
      bool ok = wait_or_abort(q_full, 0, abort_flag, p.err);
      for (int j = 0; ok && j < nlive; ++j) ok = issue_qk(j);
    }
  } else if (warp == 7) {
    if (lane == 0 && nlive > 0) {
      // ---------------- PV issuer (one thread): PV(t) once the softmax has
      // written P(t), so the QK issuer never waits behind it
      constexpr uint32_t IDESC_PV = idesc_bf16_m128(D, false, true);
      auto issue_pv = [&](int t) -> bool {
        const int s = t % STAGES;
        if (!wait_or_abort(&p_full[t & 1], (t >> 1) & 1, abort_flag, p.err)) return false;
        if (!wait_or_abort(&v_full[s], (t / STAGES) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // A = P from TMEM (row r in lane r, 16 keys = 8 columns per step)
          const uint64_t bdesc = sw128_desc(smem_addr(sV + s * C::KV_BYTES) + kk * 2048, BN * 128, 1024);
          mma_bf16_tmem_a(tmem + C::TMEM_O, tmem + C::TMEM_S + (t & 1) * BN + kk * 8, bdesc, IDESC_PV,
                          (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&v_empty[s]);
        mma_commit(&o_done[t & 1]);
        return true;
      };
      bool ok = true;
      for (int t = 0; ok && t < nlive; ++t) ok = issue_pv(t);
      // every PV has completed, and with it every QK (PV(t) follows P(t),
      // which follows S(t))
      if (ok) mma_commit(o_last);
    }
  } else {
    // ---------------- softmax warps (0-3): thread tid owns row tid (TMEM lane tid)
    const int row = tid;
    const int rq = r_tile + row;   // row of the question
    const int tok = rq / G, g = rq % G;
    const bool row_ok = rq < n_rows;
    const int lim = n_cached + tok + 1;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    {
      // this row's q (hi and lo parts) into TMEM: rows past the tile's tokens
      // and heads are zero
      const size_t qrow = ((size_t)b * p.n_kv + h) * p.t_len * G + rq;
      const uint4* qh = reinterpret_cast<const uint4*>(p.q_hi + qrow * D);
      const uint4* ql = reinterpret_cast<const uint4*>(p.q_lo + qrow * D);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint4* src = part ? ql : qh;
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {   // 32 columns = 64 bf16 = 8 x 16 bytes
          float v[32];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 u = row_ok ? src[c0 / 4 + j] : make_uint4(0, 0, 0, 0);
            v[4 * j + 0] = __uint_as_float(u.x);
            v[4 * j + 1] = __uint_as_float(u.y);
            v[4 * j + 2] = __uint_as_float(u.z);
            v[4 * j + 3] = __uint_as_float(u.w);
          }
          tmem_st32(lane_base + (part ? C::TMEM_QL : C::TMEM_QH) + c0, v);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_full);
    }
    bool ok = true;
    int tcur = next_live(0);   // key tile of the j-th live tile
    for (int j = 0; j < nlive; ++j, tcur = next_live(tcur + 1)) {
      const uint32_t sbuf = lane_base + C::TMEM_S + (j & 1) * BN;   // S(j), then P(j)
      if (!__all_sync(0xffffffffu, wait_or_abort(&s_full[j & 1], (j >> 1) & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[BN];
      {
        float t[BN / 32][32];
#pragma unroll
        for (int q4 = 0; q4 < BN / 32; ++q4) tmem_ld32(sbuf + q4 * 32, t[q4]);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < BN / 32; ++q4)
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[q4 * 32 + c] = t[q4][c];
      }
      const int key0 = kb + tcur * BN;
      // keys [key0, key0 + nvis) pass the causal / split bounds of this row;
      // under the anchor mask a document row sees all of an anchor tile
      const bool doc_anchor = anchor_docs && tok < p.n_doc;
      const int nvis = row_ok ? min(min(ke, doc_anchor && key0 >= p.n_doc ? ke : lim) - key0, BN) : 0;
      float mraw = -INFINITY;   // max of the raw scores (the scale is positive)
      if (mode == kMaskStructured && tok >= p.n_doc && key0 < p.n_doc) {
        // slot rows over document keys (slot keys are a causal prefix, and
        // document rows are causal)
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const bool vis = c < nvis && tc_structured_visible(p, tok, key0 + c);
          sv[c] = vis ? sv[c] : -INFINITY;
          mraw = fmaxf(mraw, sv[c]);
        }
      } else if (doc_anchor && key0 < p.n_doc && key0 + BN > p.n_doc) {
        // a document row's view of the tile holding the last document keys
        // and the first anchors: its causal prefix, then the anchors
        const int nend = row_ok ? min(ke - key0, BN) : 0;   // keys before the split's end
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int key = key0 + c;
          const bool vis = c < nend && (key <= tok || key >= p.n_doc);
          sv[c] = vis ? sv[c] : -INFINITY;
          mraw = fmaxf(mraw, sv[c]);
        }
      } else if (nvis >= BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c) mraw = fmaxf(mraw, sv[c]);
      } else {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          sv[c] = c < nvis ? sv[c] : -INFINITY;
          mraw = fmaxf(mraw, sv[c]);
        }
      }
      const float mt_ = mraw * p.scale_log2;   // log2 units; -inf stays -inf
      float alpha = 1.f;
      bool rescale = false;
      if (mt_ > m_run) {
        if (m_run == -INFINITY) {
          m_run = mt_;   // nothing accumulated yet for this row: O holds zeros
        } else if (mt_ - m_run > kRescaleLog2) {
          alpha = exp2f(m_run - mt_);
          m_run = mt_;
          rescale = true;
        }
      }
      const float mu = (m_run == -INFINITY) ? 0.f : m_run;
      // p = 2^(s * scale - mu): one FFMA and one ex2 per score (masked scores
      // are -inf and give 0)
      const float sc = p.scale_log2;
      float lsum0 = 0.f, lsum1 = 0.f;
      uint32_t pk[BN / 2];   // packed in place of sv as it is consumed
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float p0 = ex2_approx(fmaf(sv[c], sc, -mu)), p1 = ex2_approx(fmaf(sv[c + 1], sc, -mu));
        lsum0 += p0;
        lsum1 += p1;
        pk[c / 2] = pack2(p0, p1);
      }
      const float lsum = lsum0 + lsum1;
      l_run = l_run * alpha + lsum;
      // O rescale needs PV(j-1) finished; the warp shares the TMEM access, so
      // the whole warp takes the path when any of its rows needs it.
      if (__any_sync(0xffffffffu, rescale)) {
        if (!__all_sync(0xffffffffu, wait_or_abort(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(lane_base + C::TMEM_O + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] *= alpha;
          tmem_st32(lane_base + C::TMEM_O + c0, o);
        }
        tmem_wait_st();
      }
      // P(j) over S(j) (read above), row = lane, keys 2c and 2c + 1 in column c
#pragma unroll
      for (int c0 = 0; c0 < BN / 2; c0 += 32) {
        float v[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(pk[c0 + c]);
        tmem_st32(sbuf + c0, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
    }

    // ---------------- epilogue: the last PV must be complete before O is read
    ok = __all_sync(0xffffffffu, ok);
    if (ok && nlive > 0 && !__all_sync(0xffffffffu, wait_or_abort(o_last, 0, abort_flag, p.err)))
      ok = false;
    if (ok && nlive > 0) tc_fence_after();
    if (p.num_splits == 1) {
      const float invl = (l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        if (ok && nlive > 0) {
          tmem_ld32(lane_base + C::TMEM_O + c0, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0.f;
        }
        if (!row_ok) continue;
        __nv_bfloat16* dst = p.out + (((size_t)b * p.t_len + tok) * p.n_q + h * G + g) * D + c0;
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = o[c + e] * invl;
          *reinterpret_cast<uint4*>(dst + c) = pack8(f);
        }
      }
    }
  }

  // ---------------- teardown of the pipeline
  tc_fence_before();
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  if (aborted) {
    // let TMA copies in flight land before the shared memory is reused
    if (tid == 0) {   // the last STAGES loads of each ring (nothing is issued without live tiles)
      for (int r = 0; r < 2; ++r) {
        const int n = r ? *v_issued : *k_issued;
        uint64_t* full = r ? v_full : k_full;
        for (int jj = max(0, n - STAGES); jj < n; ++jj) mbar_wait(&full[jj % STAGES], (jj / STAGES) & 1);
      }
    }
    __syncthreads();
  }
  const int S = p.num_splits;
  float* ost = reinterpret_cast<float*>(smem + C::OFF_OST);   // [BM][D], chunk c of row r at c ^ (r & 7)
  float* mls = reinterpret_cast<float*>(smem + C::OFF_ML);    // [BM][2]
  if (S > 1 && warp < 4) {
    // Stage this split's rows: every MMA has completed (o_last) and every
    // issued K/V copy has been consumed, so the K ring is free.
    const int row = tid;
    const bool have = !aborted && nlive > 0;   // uniform over the CTA
    if (have) tc_fence_after();
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float o[32];
      if (have) {
        tmem_ld32(lane_base + C::TMEM_O + c0, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = 0.f;
      }
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const int ch = (c0 + c) / 4;
        *reinterpret_cast<float4*>(ost + row * D + ((ch ^ (row & 7)) << 2)) =
            make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
      }
    }
    mls[row * 2 + 0] = have ? m_run : -INFINITY;
    mls[row * 2 + 1] = have ? l_run : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
  }
  // That launch still completes only after this one, so the work after it
  // on the stream sees both.  (A no-op in a launch without the dependency.)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (S == 1) return;

  // ---------------- merge the S splits of the cluster; CTA r owns a row range.
  // Every CTA of the cluster reaches both cluster barriers on every path (all
  // waits above are bounded), and none leaves before the peers' reads of its
  // shared memory are done.
  cg::cluster_group cl = cg::this_cluster();
  cl.sync();
  const int rank = (int)cl.block_rank();
  const int rows_per = (BM + S - 1) / S;
  const int r0 = rank * rows_per;
  const int nr = max(0, min(BM, r0 + rows_per) - r0);
  float* sm_m = reinterpret_cast<float*>(smem + C::OFF_MRG);   // [nr][S]
  float* sm_l = sm_m + nr * S;
  float* sm_w = sm_l + nr * S;
  for (int i = tid; i < nr * S; i += kThreadsTc) {
    const int rr = i / S, sp = i % S;
    const float* peer = cl.map_shared_rank(mls, sp);
    sm_m[i] = peer[(r0 + rr) * 2 + 0];
    sm_l[i] = peer[(r0 + rr) * 2 + 1];
  }
  __syncthreads();
  for (int rr = tid; rr < nr; rr += kThreadsTc) {
    float M = -INFINITY;
    for (int sp = 0; sp < S; ++sp) M = fmaxf(M, sm_m[rr * S + sp]);
    float L = 0.f;
    for (int sp = 0; sp < S; ++sp) {
      const float ms = sm_m[rr * S + sp];
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      sm_w[rr * S + sp] = w;
      L = fmaf(sm_l[rr * S + sp], w, L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int sp = 0; sp < S; ++sp) sm_w[rr * S + sp] *= inv;
  }
  __syncthreads();
  constexpr int CH = D / 4;   // 16-byte chunks of a row
  for (int it = tid; it < nr * CH; it += kThreadsTc) {
    const int rr = it / CH, c = it % CH;
    const int row = r0 + rr;
    const int rq = r_tile + row;
    const int tok = rq / G, g = rq % G;
    if (rq >= n_rows) continue;
    const int off = row * D + ((c ^ (row & 7)) << 2);
    float4 v[kMaxClusterTc];
#pragma unroll
    for (int sp = 0; sp < kMaxClusterTc; ++sp)
      if (sp < S && sm_w[rr * S + sp] != 0.f)   // a split without keys holds no O
        v[sp] = *reinterpret_cast<const float4*>(cl.map_shared_rank(ost, sp) + off);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < kMaxClusterTc; ++sp) {
      if (sp < S && sm_w[rr * S + sp] != 0.f) {
        const float w = sm_w[rr * S + sp];
        a.x = fmaf(w, v[sp].x, a.x);
        a.y = fmaf(w, v[sp].y, a.y);
        a.z = fmaf(w, v[sp].z, a.z);
        a.w = fmaf(w, v[sp].w, a.w);
      }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y), hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p.out + (((size_t)b * p.t_len + tok) * p.n_q + h * G + g) * D + c * 4) = pk;
  }
  cl.sync();
}

template <int D, int G, bool MASKED>
KernelSetup& tc_setup() {
  static KernelSetup s;
  return s;
}

// Sets the kernel's attributes on device `dev` once (caller holds s.mu).
template <int D, int G, bool MASKED>
cudaError_t configure_tc(KernelSetup& s, int dev) {
  using C = TcCfg<D>;
  if (s.state[dev] == 0) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_tc_kernel<D, G, MASKED>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(prefill_tc_kernel<D, G, MASKED>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) cudaGetLastError();
    s.state[dev] = e == cudaSuccess ? 1 : -(int)e;
  }
  return s.state[dev] == 1 ? cudaSuccess : (cudaError_t)(-s.state[dev]);
}

template <int D, int G, bool MASKED>
cudaError_t launch_tc(const PrefillTcParams& p, cudaStream_t st) {
  using C = TcCfg<D>;
  {
    KernelSetup& s = tc_setup<D, G, MASKED>();
    const int dev = setup_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(s.mu);
    const cudaError_t e = configure_tc<D, G, MASKED>(s, dev);
    if (e != cudaSuccess) return e;
  }
  if (p.num_splits < 1 || p.num_splits > kMaxClusterTc) return cudaErrorInvalidValue;
  if (p.n_mt != (p.t_len * G + BM - 1) / BM || p.unit0 < 0 || p.n_units < 1 ||
      p.unit0 + p.n_units > p.batch * p.n_kv * p.n_mt || (int64_t)p.n_units * p.num_splits > INT32_MAX)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits * p.n_units, 1, 1);
  cfg.blockDim = dim3(kThreadsTc);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.num_splits;   // the key splits of one unit form a cluster
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.unit0 > 0) {   // the rest of the last wave, behind the launch of the units before it
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<D, G, MASKED>, p);
}

// Number of `cs`-CTA clusters of the kernel that can be resident at once
// (cached; 0 when unknown).
template <int D, int G, bool MASKED>
int tc_active_clusters(int cs) {
  using C = TcCfg<D>;
  static_assert(kMaxClusterTc < 17, "KernelSetup::clusters holds sizes up to 16");
  if (cs < 1 || cs > kMaxClusterTc) return 0;
  KernelSetup& s = tc_setup<D, G, MASKED>();
  const int dev = setup_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lk(s.mu);
  if (configure_tc<D, G, MASKED>(s, dev) != cudaSuccess) return 0;
  int* cache = s.clusters[dev];
  if (cache[cs] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(kThreadsTc);
    cfg.dynamicSmemBytes = C::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_tc_kernel<D, G, MASKED>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    cache[cs] = n > 0 ? n : -1;
  }
  return cache[cs] > 0 ? cache[cs] : 0;
}

template <int D, bool MASKED>
int active_clusters_d(int cs, int group) {
  switch (group) {
    case 1: return tc_active_clusters<D, 1, MASKED>(cs);
    case 2: return tc_active_clusters<D, 2, MASKED>(cs);
    case 4: return tc_active_clusters<D, 4, MASKED>(cs);
    case 5: return tc_active_clusters<D, 5, MASKED>(cs);
    case 8: return tc_active_clusters<D, 8, MASKED>(cs);
    default: return 0;
  }
}

template <int D, bool MASKED>
cudaError_t launch_tc_d(const PrefillTcParams& p, int group, cudaStream_t st) {
  switch (group) {
    case 1: return launch_tc<D, 1, MASKED>(p, st);
    case 2: return launch_tc<D, 2, MASKED>(p, st);
    case 4: return launch_tc<D, 4, MASKED>(p, st);
    case 5: return launch_tc<D, 5, MASKED>(p, st);
    case 8: return launch_tc<D, 8, MASKED>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

int active_clusters(int cs, int head_dim, int group, bool masked) {
  if (head_dim == 128) return masked ? active_clusters_d<128, true>(cs, group) : active_clusters_d<128, false>(cs, group);
  if (head_dim == 64) return masked ? active_clusters_d<64, true>(cs, group) : active_clusters_d<64, false>(cs, group);
  return 0;
}

}  // namespace

int prefill_tc_m_tiles(int t_len, int group) { return (t_len * group + BM - 1) / BM; }

int prefill_tc_key_tile() { return BN; }

// Key splits of each (sequence, M tile, kv head) unit: as many as keep all
// the units' clusters resident at once (one CTA per SM), at most 16 and at
// most one per key tile.  Small units counts thereby fill the SMs; with
// units >= SMs / 2 there is one split and no merge.  (Splitting units that
// run in several waves anyway, to even out the last wave, was slower: 8 x 8
// x 5 units of a 128-token G = 5 question took 336 us per layer in clusters
// of 2 against 294 us unsplit.)
void prefill_tc_plan(int units, int max_keys, int num_sms, int head_dim, int group, int* num_splits,
                     int* split_keys) {
  int s = units > 0 ? num_sms / units : 1;
  s = std::min(s, (max_keys + BN - 1) / BN);
  s = std::min(s, kMaxClusterTc);
  for (; s >= 2; --s) {
    // both instantiations take the same shared memory, so the causal one
    // answers for the masked one too; every CTA allocates all 512 TMEM
    // columns, so at most one per SM runs at a time whatever the shared
    // memory would allow (head_dim 64)
    const int n = std::min(active_clusters(s, head_dim, group, false), num_sms / s);
    if (n >= units) break;
  }
  if (s < 1) s = 1;
  int sk = (max_keys + s - 1) / s;
  sk = std::max(BN, (sk + BN - 1) / BN * BN);
  *split_keys = sk;
  *num_splits = std::max(1, (max_keys + sk - 1) / sk);
}

// Units of about equal work (`even`: a question over a longer cache) that
// fill whole waves of resident CTAs run unsplit.  The remainder of the last
// wave, when it splits (its units' clusters all resident at once), goes to
// a second launch: its keys spread over the SMs instead of a few SMs
// streaming whole units alone after the others have finished (8 x 8 x 5
// units of a 128-token G = 5 question on 152 SMs: 304 unsplit, then 16 in
// clusters of 6; 296 -> 230 us per layer).  Units of unequal work (causal
// rows over the question's own keys) stay in one launch, where the CTA
// scheduler already fills the SMs that finish early (a second launch made
// the 4000 + 1000-token extraction 2-6 % slower).
PrefillTcSchedule prefill_tc_schedule(int units, int max_keys, int num_sms, int head_dim, int group, bool even) {
  PrefillTcSchedule sc{};
  sc.bulk = units;
  prefill_tc_plan(units, max_keys, num_sms, head_dim, group, &sc.splits0, &sc.keys0);
  sc.splits1 = 1;
  sc.keys1 = sc.keys0;
  int wave = std::min(active_clusters(1, head_dim, group, false), num_sms);   // CTAs at a time (TMEM: one per SM)
  if (wave <= 0) wave = num_sms;
  if (even && sc.splits0 == 1 && units > wave && units % wave != 0) {
    const int rest = units % wave;
    int s1 = 1, k1 = 0;
    prefill_tc_plan(rest, max_keys, num_sms, head_dim, group, &s1, &k1);
    if (s1 > 1) {
      sc.bulk = units - rest;
      sc.splits1 = s1;
      sc.keys1 = k1;
    }
  }
  return sc;
}

cudaError_t launch_prefill_tc(const PrefillTcParams& p, int head_dim, int group, cudaStream_t st) {
  const bool masked = p.mask_mode != kMaskCausal;
  if (head_dim == 128) return masked ? launch_tc_d<128, true>(p, group, st) : launch_tc_d<128, false>(p, group, st);
  if (head_dim == 64) return masked ? launch_tc_d<64, true>(p, group, st) : launch_tc_d<64, false>(p, group, st);
  return cudaErrorInvalidValue;
}

}  // namespace c2kv
