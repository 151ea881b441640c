// Linear layers of the synthetic-weight decoder step on the tensor cores:
// Y[t][n] = sum_k X[t][k] W[n][k] for a few tokens t (the decode batch, or a
// question), with fused epilogues (residual add, q/k/v split, SwiGLU).
//
// C2KV explainer (paper-daily.com), section "the problem" (它到底在解决什么问题？)
// and its Fig. 1: the time to first token and the decode rate of the whole
// model are what cache reuse buys; the projections and the MLP run between
// the attention calls of every layer.
//
// With few tokens the product is weight-bandwidth-bound: each weight is read
// once and used by every token.  So weights are the MMA's M dimension (128-
// row tiles, K-major A by TMA with 128-byte swizzle) and the tokens its N
// dimension (padded to a multiple of 16, K-major B).  The (tile, 64-wide K
// chunk) work items of the whole product are laid end to end and cut into one
// equal contiguous range per CTA, one CTA per SM (the split of
// decode_plan.h, with the output tiles as units), so every SM streams the
// same share of the weights whatever the tile count.  A CTA whose range
// covers a whole tile applies the epilogue from TMEM; a partial tile is
// stored as fp32 and the CTA whose chunks complete the tile's count sums
// the partials (in CTA order: deterministic) and applies the epilogue.
//
// Roles: warps 0-3 epilogue (thread r = weight row r of the tile = TMEM lane
// r), warp 4 lane 0 TMA, warp 5 lane 0 MMA.  The weight tiles of the first
// stages are requested before the kernel waits for the previous one on the
// stream (weights do not depend on it); the activations after.
#include <float.h>

#include <algorithm>

#include <cooperative_groups.h>

#include "c2kv_internal.h"
#include "decode_plan.h"
#include "tcgen05.h"

namespace cg = cooperative_groups;

namespace c2kv {

namespace {

constexpr int LT_BM = 128;            // weight rows per tile
constexpr int LT_BK = 64;             // K elements per chunk (one 128-byte swizzle atom)
constexpr int LT_THREADS = 192;
constexpr int LT_EPI_THREADS = 128;
constexpr int LT_W_BYTES = LT_BM * LT_BK * 2;   // 16 KB
constexpr int LT_MAX_STAGES = 16;
constexpr int LT_MISC = 2 * LT_MAX_STAGES + 8;  // barriers
constexpr int LT_XCH_COLS = 16;                  // SwiGLU exchange: columns per round
constexpr int kMergeChunk = 16;                  // partial tiles whose loads are in flight together

__host__ __device__ constexpr int lt_stage_bytes(int n_pad) { return LT_W_BYTES + n_pad * LT_BK * 2; }

constexpr int kLinearMaxCtas = 512;              // CTAs of one launch (2 per SM)

struct LtLayout {
  int stage, off_xch, off_map, off_slots, off_bar, off_misc, total;
};

__host__ __device__ inline LtLayout lt_layout(int n_pad, int stages) {
  LtLayout l;
  l.stage = lt_stage_bytes(n_pad);
  l.off_xch = stages * l.stage;                                   // SwiGLU exchange [64][16] fp32
  l.off_map = l.off_xch + 64 * LT_XCH_COLS * 4;
  l.off_slots = l.off_map + (int)((sizeof(DecodeMap) + 15) / 16 * 16);   // merge: contributors' slots
  l.off_bar = l.off_slots + kLinearMaxCtas * 4;
  l.off_misc = l.off_bar + LT_MISC * 8;
  l.total = l.off_misc + 64 + 1024;                               // + slack for 1024-byte alignment
  return l;
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

template <int EPI>
__global__ void __launch_bounds__(LT_THREADS, 2) linear_tc_kernel(const __grid_constant__ LinearParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const LtLayout lay = lt_layout(p.n_pad, p.stages);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.off_bar);
  uint64_t* full = bars;                        // [stages]
  uint64_t* empty = full + LT_MAX_STAGES;       // [stages]
  uint64_t* acc_full = empty + LT_MAX_STAGES;   // [2]
  uint64_t* acc_free = acc_full + 2;            // [2]
  uint64_t* grp_bar = acc_free + 2;
  uint64_t* mma_done = grp_bar + 1;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + lay.off_misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.off_misc + 8);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + lay.off_misc + 16);
  float* xch = reinterpret_cast<float*>(smem + lay.off_xch);
  DecodeMap& M = *reinterpret_cast<DecodeMap*>(smem + lay.off_map);
  int32_t* mslots = reinterpret_cast<int32_t*>(smem + lay.off_slots);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int kc = p.k_in / LT_BK;                // chunks per tile
  const int tiles = p.n_out / LT_BM;
  // TMEM: two accumulators of n_pad columns, at columns 0 and cols / 2 of an
  // allocation of a power of two >= 32 columns
  int cols = 32;
  while (cols < 2 * p.n_pad) cols <<= 1;
  const int acc_off = cols / 2;

  if (tid == 0) {
    // one "sequence" whose units are the output tiles, kc chunks each
    const int32_t keys = kc * kDecKeyTile;
    decode_map_build(M, &keys, 1, tiles, (int)gridDim.x);
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], LT_EPI_THREADS);
    }
    mbar_init(grp_bar, 4);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr((const void*)tmem_slot)),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int64_t x0, x1;
  if (p.cs > 0) {
    // one cluster of cs CTAs per tile; CTA r of it takes an equal share of the
    // tile's chunks (the host keeps cs <= chunks, so every CTA has one)
    const int tile = cta / p.cs, r = cta % p.cs;
    x0 = (int64_t)tile * kc + (int64_t)r * kc / p.cs;
    x1 = (int64_t)tile * kc + (int64_t)(r + 1) * kc / p.cs;
  } else {
    x0 = decode_cta_first(M, cta);
    x1 = decode_cta_first(M, cta + 1);
  }
  const int nitems = (int)(x1 - x0);
  if (nitems == 0) {
    if (warp == 4)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
    return;
  }
  const int stage_bytes = lay.stage;
  int issued = 0;

  if (warp == 4) {
    if (lane == 0) {
      // ---------------- TMA producer.  The first stages' weight tiles go out
      // before the wait for the previous kernel, their activation tiles after.
      const int pre = min(p.stages, nitems);
      for (int j = 0; j < pre; ++j) {
        const int64_t x = x0 + j;
        const int tile = (int)(x / kc), ch = (int)(x % kc);
        mbar_arrive_expect_tx(&full[j], stage_bytes);
        tma_load_2d(smem + j * stage_bytes, &p.tm_w, ch * LT_BK, tile * LT_BM, &full[j]);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int j = 0; j < pre; ++j) {
        const int ch = (int)((x0 + j) % kc);
        tma_load_2d(smem + j * stage_bytes + LT_W_BYTES, &p.tm_x, ch * LT_BK, 0, &full[j]);
      }
      issued = pre;
      for (int j = pre; j < nitems; ++j) {
        const int s = j % p.stages;
        if (!wait_or_abort(&empty[s], ((j - p.stages) / p.stages) & 1, abort_flag, p.err)) break;
        const int64_t x = x0 + j;
        const int tile = (int)(x / kc), ch = (int)(x % kc);
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        tma_load_2d(smem + s * stage_bytes, &p.tm_w, ch * LT_BK, tile * LT_BM, &full[s]);
        tma_load_2d(smem + s * stage_bytes + LT_W_BYTES, &p.tm_x, ch * LT_BK, 0, &full[s]);
        ++issued;
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------- MMA issuer: one accumulator per segment (the CTA's
      // part of one tile), alternating between the two TMEM buffers
      const uint32_t idesc = idesc_bf16_m128(p.n_pad, false, false);
      bool ok = true;
      int seg = -1;
      for (int j = 0; ok && j < nitems; ++j) {
        const int64_t x = x0 + j;
        const int ch = (int)(x % kc);
        const bool first = j == 0 || ch == 0;
        const bool last = j == nitems - 1 || ch == kc - 1;
        if (first) {
          ++seg;
          if (seg >= 2) ok = wait_or_abort(&acc_free[seg & 1], ((seg - 2) >> 1) & 1, abort_flag, p.err);
        }
        const int s = j % p.stages;
        if (ok) ok = wait_or_abort(&full[s], (j / p.stages) & 1, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sw = smem_addr(smem + s * stage_bytes);
#pragma unroll
        for (int kk = 0; kk < LT_BK / 16; ++kk) {
          const uint64_t a = sw128_desc(sw + kk * 32, 16, 1024);
          const uint64_t b = sw128_desc(sw + LT_W_BYTES + kk * 32, 16, 1024);
          mma_bf16(tmem + (seg & 1) * acc_off, a, b, idesc, (!first || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
        if (last) mma_commit(&acc_full[seg & 1]);
      }
      mma_commit(mma_done);
      mbar_wait(mma_done, 0);
    }
  } else if (warp < 4) {
    // ---------------- epilogue: thread tid owns weight row tid of each tile
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int T = p.tokens;
    int k_sync = 0, seg = 0, arrived = -1;
    bool ok = true;
    // Stores one output column chunk: v[c] is token c0 + c of weight row n.
    // (loops over the 16 columns are unrolled with a guard so that v stays in
    // registers)
    auto emit = [&](int tile, int c0, const float (&v)[16], int nc) {
      const int n = tile * LT_BM + tid;
      if (EPI == kLinearSwiglu) {
        // rows 0..63 of the tile are gate rows of features 64*tile + r, rows
        // 64..127 the up rows of the same features
        if (tid >= 64) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (c < nc) xch[(tid - 64) * LT_XCH_COLS + c] = v[c];
        }
        return;
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int t = c0 + c;
        if (c >= nc) break;
        float val = v[c];
        if (EPI == kLinearAdd) val += __bfloat162float(p.residual[(size_t)t * p.n_out + n]);
        if (EPI == kLinearSplit3) {
          if (n < p.split1)
            p.y[(size_t)t * p.split1 + n] = __float2bfloat16_rn(val);
          else if (n < p.split2)
            p.y2[(size_t)t * (p.split2 - p.split1) + (n - p.split1)] = __float2bfloat16_rn(val);
          else
            p.y3[(size_t)t * (p.n_out - p.split2) + (n - p.split2)] = __float2bfloat16_rn(val);
        } else {
          p.y[(size_t)t * p.n_out + n] = __float2bfloat16_rn(val);
        }
      }
    };
    // SwiGLU: after the up rows staged their values, the gate rows finish.
    auto emit_swiglu = [&](int tile, int c0, const float (&v)[16], int nc) -> bool {
      if (!group_sync(grp_bar, k_sync, abort_flag, p.err)) return false;
      if (tid < 64) {
        const int f = tile * 64 + tid;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int t = c0 + c;
          if (c >= nc) break;
          p.y[(size_t)t * (p.n_out / 2) + f] = __float2bfloat16_rn(silu(v[c]) * xch[tid * LT_XCH_COLS + c]);
        }
      }
      return group_sync(grp_bar, k_sync, abort_flag, p.err);   // xch free again
    };
    DecodeTile d = decode_locate(M, x0);
    for (int j0 = 0; ok && j0 < nitems; ++seg) {
      const int tile = d.h, ch0 = d.t;
      const int n = min(kc - ch0, nitems - j0);
      const bool whole = ch0 == 0 && n == kc;
      const int buf = seg & 1;
      if (!__all_sync(0xffffffffu, wait_or_abort(&acc_full[buf], (seg >> 1) & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int slot = 2 * cta + (seg == 0 ? 0 : 1);
      // Column chunks of 16 tokens: whole tiles go to the epilogue, partial
      // ones to this CTA's slot.
      for (int c0 = 0; ok && c0 < T; c0 += 16) {
        float v[16];
        tmem_ld_cols<16>(lane_base + buf * acc_off + c0, v);
        tmem_wait_ld();
        const int nc = min(16, T - c0);
        if (whole) {
          emit(tile, c0, v, nc);
          if (EPI == kLinearSwiglu) ok = emit_swiglu(tile, c0, v, nc);
        } else {
          if (p.cs > 1) {
            // this CTA's share of a cluster-split tile, staged in its own
            // shared memory ([n_pad][128] fp32 over the ring: every MMA has
            // completed) for the cluster's reduction after the teardown
            float* cpart = reinterpret_cast<float*>(smem);
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c < nc) cpart[(c0 + c) * LT_BM + tid] = v[c];
          } else {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c < nc) p.part[((size_t)slot * p.n_pad + c0 + c) * LT_BM + tid] = v[c];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_free[buf]);
      if (ok && !whole && p.cs == 0) {
        // every partial store of the CTA is ordered before tid 0's arrival
        ok = group_sync(grp_bar, k_sync, abort_flag, p.err);
        if (ok && tid == 0) {
          int prev;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                       : "=r"(prev)
                       : "l"(p.counters + tile), "r"(n)
                       : "memory");
          const bool lastc = prev + n == kc;
          if (lastc) p.counters[tile] = 0;   // every CTA of the tile has arrived
          *last_flag = lastc ? 1 : 0;
          arrived = seg;
        }
        if (ok) ok = group_sync(grp_bar, k_sync, abort_flag, p.err);
        if (ok && *last_flag) {
          // ---- sum the tile's partials in CTA order, then the epilogue
          const int64_t uf = (int64_t)tile * kc;
          const int cf = decode_cta_of(M, uf), cl = decode_cta_of(M, uf + kc - 1);
          const int nctr = cl - cf + 1;
          // the contributors' slots, one per thread (each takes a few 64-bit
          // divisions), then kMergeChunk contributors' loads in flight at a
          // time, summed in CTA order
          for (int kk = tid; kk < nctr; kk += LT_EPI_THREADS)
            mslots[kk] = decode_cta_empty(M, cf + kk) ? -1 : decode_slot_of(M, cf + kk, uf);
          ok = group_sync(grp_bar, k_sync, abort_flag, p.err);
          for (int c0 = 0; ok && c0 < T; c0 += 16) {
            const int nc = min(16, T - c0);
            float v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = 0.f;
            for (int q0 = 0; q0 < nc; q0 += 4) {   // 4 columns at a time
              for (int k0 = 0; k0 < nctr; k0 += kMergeChunk) {
                float got[kMergeChunk][4];
#pragma unroll
                for (int k = 0; k < kMergeChunk; ++k) {
                  const int sl = k0 + k < nctr ? mslots[k0 + k] : -1;   // -1: an empty CTA
                  const float* src = p.part + ((size_t)(sl < 0 ? 0 : sl) * p.n_pad + c0 + q0) * LT_BM + tid;
#pragma unroll
                  for (int cc = 0; cc < 4; ++cc)
                    got[k][cc] = (sl >= 0 && q0 + cc < nc) ? __ldcg(src + (size_t)cc * LT_BM) : 0.f;
                }
#pragma unroll
                for (int k = 0; k < kMergeChunk; ++k)
#pragma unroll
                  for (int cc = 0; cc < 4; ++cc) v[q0 + cc] += got[k][cc];
              }
            }
            emit(tile, c0, v, nc);
            if (EPI == kLinearSwiglu) ok = emit_swiglu(tile, c0, v, nc);
          }
        }
      }
      j0 += n;
      if (j0 < nitems) d = decode_locate(M, x0 + j0);
    }
    if (!ok && tid == 0 && p.cs == 0) {
      // gave up: add the remaining partial tiles' chunks to their counters
      // (their outputs are undefined) so every counter ends at zero
      DecodeTile e = decode_locate(M, x0);
      int sg = 0;
      for (int j0 = 0; j0 < nitems; ++sg) {
        const int n = min(kc - e.t, nitems - j0);
        if (sg > arrived && !(e.t == 0 && n == kc)) {
          const int prev = atomicAdd(p.counters + e.h, n);
          if (prev + n == kc) p.counters[e.h] = 0;
        }
        j0 += n;
        if (j0 < nitems) e = decode_locate(M, x0 + j0);
      }
    }
  }

  // ---------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 4 && lane == 0) {
    for (int j = max(0, issued - p.stages); j < issued; ++j) mbar_wait(&full[j % p.stages], (j / p.stages) & 1);
  }
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
  }
  if (p.cs > 1) {
    // ---------------- the cluster's reduction: CTA r sums its share of the
    // tile's rows (SwiGLU: its share of the gate/up row pairs) over the cs
    // staged partials, in rank order, and applies the epilogue.  Every CTA
    // reaches both cluster barriers on every path (all waits above are
    // bounded), and none leaves before its peers' reads are done.
    cg::cluster_group clu = cg::this_cluster();
    clu.sync();
    const int cs = p.cs, r = (int)clu.block_rank(), tile = cta / cs;
    const int T = p.tokens;
    const float* cpart = reinterpret_cast<const float*>(smem);
    const float* peer[8];
#pragma unroll
    for (int sp = 0; sp < 8; ++sp) peer[sp] = sp < cs ? clu.map_shared_rank(cpart, sp) : cpart;
    auto tile_sum = [&](int t, int row) {
      float v = 0.f;
#pragma unroll
      for (int sp = 0; sp < 8; ++sp)
        if (sp < cs) v += peer[sp][t * LT_BM + row];
      return v;
    };
    if (EPI == kLinearSwiglu) {
      const int fp = (LT_BM / 2 + cs - 1) / cs, f0 = r * fp, nf = max(0, min(LT_BM / 2, f0 + fp) - f0);
      for (int it = tid; it < nf * T; it += LT_THREADS) {
        const int t = it / nf, f = f0 + it % nf;
        const float gt = tile_sum(t, f), up = tile_sum(t, f + LT_BM / 2);
        p.y[(size_t)t * (p.n_out / 2) + tile * (LT_BM / 2) + f] = __float2bfloat16_rn(silu(gt) * up);
      }
    } else {
      const int rp = (LT_BM + cs - 1) / cs, r0 = r * rp, nr = max(0, min(LT_BM, r0 + rp) - r0);
      for (int it = tid; it < nr * T; it += LT_THREADS) {
        const int t = it / nr, row = r0 + it % nr, n = tile * LT_BM + row;
        float val = tile_sum(t, row);
        if (EPI == kLinearAdd) val += __bfloat162float(p.residual[(size_t)t * p.n_out + n]);
        if (EPI == kLinearSplit3) {
          if (n < p.split1)
            p.y[(size_t)t * p.split1 + n] = __float2bfloat16_rn(val);
          else if (n < p.split2)
            p.y2[(size_t)t * (p.split2 - p.split1) + (n - p.split1)] = __float2bfloat16_rn(val);
          else
            p.y3[(size_t)t * (p.n_out - p.split2) + (n - p.split2)] = __float2bfloat16_rn(val);
        } else {
          p.y[(size_t)t * p.n_out + n] = __float2bfloat16_rn(val);
        }
      }
    }
    clu.sync();
  }
}

// ---------------------------------------------------------------------------
// RMSNorm of `tokens` rows of `dim`: y = x / sqrt(mean(x^2) + eps) * w, with
// the sum of squares in fp32.  One CTA per row.
// ---------------------------------------------------------------------------
__global__ void rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
                               __nv_bfloat16* __restrict__ y, int dim, float eps) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float part[32];
  const int row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * dim);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  uint4* yr = reinterpret_cast<uint4*>(y + (size_t)row * dim);
  const int n8 = dim / 8;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n8; i += blockDim.x) {
    float f[8];
    unpack8(xr[i], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) part[0] = v;
  }
  __syncthreads();
  const float inv = rsqrtf(part[0] / (float)dim + eps);
  for (int i = threadIdx.x; i < n8; i += blockDim.x) {
    float f[8], g[8];
    unpack8(xr[i], f);
    unpack8(wr[i], g);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = f[e] * inv * g[e];
    yr[i] = pack8(f);
  }
}

template <int EPI>
KernelSetup& lt_setup() {
  static KernelSetup s;
  return s;
}

template <int EPI>
cudaError_t launch_lt(const LinearParams& p, int ctas, bool overlap, cudaStream_t st) {
  const int smem = lt_layout(p.n_pad, p.stages).total;
  {
    KernelSetup& s = lt_setup<EPI>();
    const int dev = setup_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(s.mu);
    if (s.state[dev] == 0) {
      const cudaError_t e =
          cudaFuncSetAttribute(linear_tc_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLinearSmemMax);
      if (e != cudaSuccess) cudaGetLastError();
      s.state[dev] = e == cudaSuccess ? 1 : -(int)e;
    }
    if (s.state[dev] != 1) return (cudaError_t)(-s.state[dev]);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(LT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.cs > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p.cs;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, linear_tc_kernel<EPI>, p);
}

}  // namespace

// Pipeline depth for `n_pad` token columns: as deep as half an SM's shared
// memory allows, so that two CTAs fit on an SM and a launch's CTAs become
// resident, and stream their first weight tiles, while the kernel before it
// on the stream finishes.  (A decode-time product moves ~44 GB/s per SM;
// ~100 KB in flight covers the ~2 us memory latency.)
int linear_stages(int n_pad) {
  int s = LT_MAX_STAGES;
  while (s > 2 && lt_layout(n_pad, s).total > kLinearSmemPerCta) --s;
  return s;
}

// The split of a product: with at most as many tiles as the launch has CTAs
// (two per SM), one cluster of cs CTAs per tile, cs the largest power of two
// up to 8 with cs * tiles CTAs and at most one CTA per chunk, so that a
// tile's partials are summed in distributed shared memory instead of through
// global memory; cs = 1 when every CTA can own a whole tile.  (Clusters of 6
// for the 48 tiles of the fused QKV projection took 20.5 us against 14.0 us
// in clusters of 4.)  With more tiles, or a staged partial larger than the
// shared-memory ring, 0: the even split over all CTAs.
int linear_plan_cs(int n_out, int k_in, int n_pad, int ctas_max) {
  const int tiles = n_out / LT_BM, kc = k_in / LT_BK;
  if (tiles < 1 || tiles > ctas_max) return 0;
  int cs = 1;
  while (cs < 8 && 2 * cs * tiles <= ctas_max && 2 * cs <= kc) cs *= 2;
  const int stages = linear_stages(n_pad);
  if (cs > 1 && n_pad * LT_BM * 4 > stages * lt_stage_bytes(n_pad)) return 0;
  return cs;
}

cudaError_t launch_linear(const LinearParams& p, int ctas, bool overlap, cudaStream_t st) {
  if (p.stages < 2 || p.stages > LT_MAX_STAGES || lt_layout(p.n_pad, p.stages).total > kLinearSmemMax)
    return cudaErrorInvalidValue;
  if (p.cs < 0 || p.cs > 8) return cudaErrorInvalidValue;
  if (p.cs > 0 && (ctas != (p.n_out / LT_BM) * p.cs || p.cs > p.k_in / LT_BK ||
                   (p.cs > 1 && p.n_pad * LT_BM * 4 > p.stages * lt_stage_bytes(p.n_pad))))
    return cudaErrorInvalidValue;
  switch (p.epi) {
    case kLinearStore: return launch_lt<kLinearStore>(p, ctas, overlap, st);
    case kLinearAdd: return launch_lt<kLinearAdd>(p, ctas, overlap, st);
    case kLinearSplit3: return launch_lt<kLinearSplit3>(p, ctas, overlap, st);
    case kLinearSwiglu: return launch_lt<kLinearSwiglu>(p, ctas, overlap, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const __nv_bfloat16* w, __nv_bfloat16* y, int tokens, int dim,
                           float eps, bool overlap, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tokens);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, x, w, y, dim, eps);
}

}  // namespace c2kv
