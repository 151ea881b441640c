// Composition of stored segments into the cache (host-link gather with
// re-rotation), and rotate-and-append of new tokens.
//
// C2KV explainer (paper-daily.com), section "positions at concatenation"
// (拼接时位置怎么处理？): segments are stored before RoPE and rotated at
// composition time; slot j of composed document c sits at
// off_c + min((j+1)k, n_c) - 1, where off_c is the summed original length of
// the documents before it.  Rotation is the rotate-half form: pair
// (i, i + d/2) turns by pos * theta^(-2i/d).
#include <algorithm>

#include "c2kv_internal.h"

namespace c2kv {

namespace {

// ---------------------------------------------------------------------------
// Per-row cos/sin table: for every cache row r, the d/2 angles of its
// position as fp32 hi/lo pairs of the fp64 sincos.  Composed mode: rows below
// n_total are composed slots (slot j of composed document c at
// off_c + min((j+1)k, n_c) - 1, found by binary search over the segment
// table); later rows are the appended question and answer tokens at
// l_tot + (r - n_total).  Explicit mode reads positions from pos_in;
// extraction mode puts n_doc document tokens at 0..n_doc-1 and slot s at
// min((s+1)k, n_doc) - 1.  One thread per (row, frequency).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int table_position(const TableParams& p, int r) {
  if (p.mode == kTableExplicit) return p.pos_in[r];
  if (p.mode == kTableExtraction) return r < p.n_doc ? r : min((r - p.n_doc + 1) * p.kblk, p.n_doc) - 1;
  if (r >= p.n_total) return p.l_tot + (r - p.n_total);
  int lo = 0, hi = p.n_docs - 1;   // last segment with seg.slot0 <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seg[mid].slot0 <= r) lo = mid; else hi = mid - 1;
  }
  const SegDesc sd = p.seg[lo];
  return sd.off + min((r - sd.slot0 + 1) * p.k, sd.n_tokens) - 1;
}

__global__ void rope_table_kernel(const __grid_constant__ TableParams p) {
  const int total = p.rows * p.half;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int r = i / p.half, f = i % p.half;
    const int pos = table_position(p, r);
    if (f == 0 && p.pos_out != nullptr) p.pos_out[r] = pos;
    p.tab[i] = rope_cos_sin2(pos, p.inv_freq[f]);
  }
}

// ---------------------------------------------------------------------------
// K0 + K1: the composition of one request over a range of layers, in one
// pass from the pinned host pool to the cache.  The SMs read each
// document's pre-RoPE K and V rows straight from the pinned pool (mapped
// into the device's address space) over the host link, rotate K at the
// slot's composed position and write K and V at their composed rows.  (A
// copy-engine transfer followed by an in-place rotation reads and writes K
// in HBM once more, and needs one 2-D copy per document and layer group;
// the 16-byte loads of a few CTAs saturate the link on their own.)
//
// A few persistent CTAs (kComposeCtas): enough loads in flight to cover the
// link's latency, and a footprint small enough to sit beside the decode
// kernel of another request on the same SMs (its registers and shared
// memory fit beside the decode kernel's for up to 5 q heads per kv head).
// A CTA takes tiles of kSlots (8) consecutive composed slots in turn: it
// stages their rows of the cos/sin table in shared memory once (transposed,
// pair 8c + e at e * TPR + c, so that the 8 lanes of a row read 8
// neighbouring entries), looks up each slot's document and index in it,
// then moves the slots' rows of every (layer, kv head) of the range.  A
// thread owns the 8 pairs of one 16-byte chunk of K (and the same chunks of
// V).
// ---------------------------------------------------------------------------
constexpr int kSlots = 8;
constexpr int kComposeThreads = 128;

template <int D>
__global__ void __launch_bounds__(kComposeThreads) compose_kernel(const __grid_constant__ ComposeParams p) {
  constexpr int H = D / 2;
  constexpr int TPR = H / 8;   // threads per row, each owns 8 pairs
  __shared__ CosSin2 tab[kSlots][H];
  __shared__ const __nv_bfloat16* src_k[kSlots];   // the slot's row in layer 0, kv head 0 of its document
  __shared__ const __nv_bfloat16* src_v[kSlots];
  __shared__ int64_t src_lh[kSlots];               // elements between (layer, head) runs of its document

  const int n_tiles = (p.n_total + kSlots - 1) / kSlots;
  const int n_rows = (p.layer1 - p.layer0) * p.n_kv;   // (layer, head) row blocks
  const int work = n_rows * kSlots * TPR;
  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int slot0 = tile * kSlots;
    const int n_here = min(kSlots, p.n_total - slot0);
    __syncthreads();   // the previous tile's staged rows are no longer read
    for (int i = threadIdx.x; i < n_here * H; i += kComposeThreads) {
      const int f = i % H;
      tab[i / H][(f % 8) * TPR + f / 8] = p.tab[(size_t)slot0 * H + i];
    }
    if (threadIdx.x < n_here) {
      const int s = slot0 + threadIdx.x;
      int lo = 0, hi = p.n_docs - 1;   // last document with seg.slot0 <= s
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].slot0 <= s) lo = mid; else hi = mid - 1;
      }
      const ComposeSeg sg = p.seg[lo];
      const int64_t lh = (int64_t)sg.n_slots * D;
      const int64_t off = (int64_t)p.layer0 * p.n_kv * lh + (int64_t)(s - sg.slot0) * D;
      src_k[threadIdx.x] = sg.k + off;
      src_v[threadIdx.x] = sg.v + off;
      src_lh[threadIdx.x] = lh;
    }
    __syncthreads();

    constexpr int U = 4;
    for (int w0 = threadIdx.x; w0 < work; w0 += kComposeThreads * U) {
      uint4 ka[U], kb[U], va[U], vb[U];
      int r_[U], c_[U];
      size_t dst[U];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int w = w0 + u * kComposeThreads;
        const int c = w % TPR;
        const int r = (w / TPR) % kSlots;
        const int lh = w / (TPR * kSlots);
        ok[u] = (w < work) && (r < n_here);
        r_[u] = r;
        c_[u] = c;
        dst[u] = ((size_t)(p.layer0 * p.n_kv + lh) * p.cap + slot0 + r) * D;
        if (ok[u]) {
          const uint4* ks = reinterpret_cast<const uint4*>(src_k[r] + lh * src_lh[r]);
          const uint4* vs = reinterpret_cast<const uint4*>(src_v[r] + lh * src_lh[r]);
          ka[u] = ks[c];
          kb[u] = ks[c + TPR];
          va[u] = vs[c];
          vb[u] = vs[c + TPR];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (ok[u]) {
          rotate8_df<TPR>(ka[u], kb[u], &tab[r_[u]][c_[u]]);
          uint4* kd = reinterpret_cast<uint4*>(p.k_cache + dst[u]);
          uint4* vd = reinterpret_cast<uint4*>(p.v_cache + dst[u]);
          kd[c_[u]] = ka[u];
          kd[c_[u] + TPR] = kb[u];
          vd[c_[u]] = va[u];
          vd[c_[u] + TPR] = vb[u];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// K4: rotate t_len new keys per sequence and append them (with their values)
// at rows row0 + i of the cache, rotating with the table row of that cache
// row.  Threads past the kv heads rotate q into the tensor-core tile layout.
// grid (t_len, batch), one thread per (head, 8-pair chunk).
// ---------------------------------------------------------------------------
template <int D>
__global__ void append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int H = D / 2;
  constexpr int TPR = H / 8;
  __shared__ CosSin2 tab[H];
  const int i = blockIdx.x;
  const int b = blockIdx.y;
  const int row0 = p.row_d ? p.row_d[b] : p.row_h[b];
  if (row0 < 0 || row0 + p.t_len > p.cap) {
    if (threadIdx.x == 0 && i == 0) atomicOr(p.err, kErrLength);
    return;
  }
  for (int f = threadIdx.x; f < H; f += blockDim.x) tab[f] = p.tab[b][(size_t)(row0 + i) * H + f];
  __syncthreads();
  const int h = threadIdx.x / TPR;
  const int c = threadIdx.x % TPR;
  if (h >= p.n_kv) {
    const int hq = h - p.n_kv;
    if (p.q_src == nullptr || hq >= p.n_q) return;
    const int grp = p.n_q / p.n_kv;
    const uint4* qs = reinterpret_cast<const uint4*>(p.q_src + (((size_t)b * p.t_len + i) * p.n_q + hq) * D);
    // q as two bf16 parts: hi, the correctly rounded rotation, and lo, the
    // rounded rest (hi + lo is within ~2^-16 of the exact rotation)
    float x[8], y[8];
    unpack8(qs[c], x);
    unpack8(qs[c + TPR], y);
    uint32_t h0[8], l0[8], h1[8], l1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const CosSin2 t = tab[c * 8 + e];
      float hi, lo;
      dot2_df(x[e], t.ch, t.cl, -y[e], t.sh, t.sl, hi, lo);   // x cos - y sin
      h0[e] = df_to_bf16_bits(hi, lo);
      l0[e] = bf16_bits_rn(__fadd_rn(__fsub_rn(hi, __uint_as_float(h0[e] << 16)), lo));
      dot2_df(y[e], t.ch, t.cl, x[e], t.sh, t.sl, hi, lo);    // y cos + x sin
      h1[e] = df_to_bf16_bits(hi, lo);
      l1[e] = bf16_bits_rn(__fadd_rn(__fsub_rn(hi, __uint_as_float(h1[e] << 16)), lo));
    }
    const size_t qoff = ((((size_t)b * p.n_kv + hq / grp) * p.t_len + i) * grp + hq % grp) * D;
    uint4* qd = reinterpret_cast<uint4*>(p.q_dst + qoff);
    uint4* ql = reinterpret_cast<uint4*>(p.q_dst_lo + qoff);
    qd[c] = pack_bits8(h0);
    qd[c + TPR] = pack_bits8(h1);
    ql[c] = pack_bits8(l0);
    ql[c + TPR] = pack_bits8(l1);
    return;
  }
  const size_t src = (((size_t)b * p.t_len + i) * p.n_kv + h) * D;
  const size_t dst = ((size_t)h * p.cap + row0 + i) * D;
  const uint4* ks = reinterpret_cast<const uint4*>(p.k_src + src);
  const uint4* vs = reinterpret_cast<const uint4*>(p.v_src + src);
  uint4 a = ks[c], bb = ks[c + TPR];
  rotate8_df(a, bb, &tab[c * 8]);
  uint4* kd = reinterpret_cast<uint4*>(p.k_dst[b] + dst);
  uint4* vd = reinterpret_cast<uint4*>(p.v_dst[b] + dst);
  kd[c] = a;
  kd[c + TPR] = bb;
  vd[c] = vs[c];
  vd[c + TPR] = vs[c + TPR];
}

__global__ void advance_kernel(int batch, int32_t* n_cached, int delta) {
  const int b = threadIdx.x;
  if (b < batch) n_cached[b] += delta;
}

}  // namespace

cudaError_t launch_compose(const ComposeParams& p, int head_dim, cudaStream_t st) {
  const int blocks = std::min(kComposeCtas, (p.n_total + kSlots - 1) / kSlots);
  if (blocks == 0) return cudaSuccess;
  if (head_dim == 128) compose_kernel<128><<<blocks, kComposeThreads, 0, st>>>(p);
  else compose_kernel<64><<<blocks, kComposeThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams& p, int head_dim, int batch, cudaStream_t st) {
  const dim3 grid(p.t_len, batch);
  const int threads = (p.n_kv + (p.q_src ? p.n_q : 0)) * (head_dim / 16);
  if (head_dim == 128) append_kernel<128><<<grid, threads, 0, st>>>(p);
  else append_kernel<64><<<grid, threads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_advance(int batch, int32_t* n_cached, int delta, cudaStream_t st) {
  advance_kernel<<<1, 32, 0, st>>>(batch, n_cached, delta);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(const TableParams& p, cudaStream_t st) {
  const int total = p.rows * p.half;
  if (total == 0) return cudaSuccess;
  const int blocks = (total + 255) / 256;
  rope_table_kernel<<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace c2kv
