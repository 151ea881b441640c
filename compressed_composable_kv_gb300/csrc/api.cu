// C ABI of the C2KV composed-cache path: pinned segment store, composition
// (host->device streaming + re-rotation), and the attention entry points.
// Every argument check happens here, on the host, before anything is
// enqueued.  See include/c2kv.h for the contract of each call.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include <cudaTypedefs.h>

#include "c2kv_internal.h"
#include "decode_plan.h"

using namespace c2kv;

namespace {

thread_local std::string g_err;

c2kv_status fail(c2kv_status st, const std::string& msg) {
  g_err = msg;
  return st;
}

#define C2KV_CUDA(call)                                                                   \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return fail(C2KV_ECUDA, std::string(#call) + ": " + cudaGetErrorString(e_));        \
  } while (0)

// Kernel launches enqueued by this library (c2kv_kernel_launches).
std::atomic<uint64_t> g_kernel_launches{0};

#define C2KV_LAUNCH(call)                                             \
  do {                                                                \
    C2KV_CUDA(call);                                                  \
    g_kernel_launches.fetch_add(1, std::memory_order_relaxed);        \
  } while (0)

// Device error word, one per device that loads the library.
__device__ unsigned int g_error_word = 0;

constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::mutex g_dev_mu;

c2kv_status device_state(unsigned** err, int* num_sms) {
  int dev = 0;
  C2KV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(C2KV_EINVAL, "device index out of range");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    C2KV_CUDA(cudaGetSymbolAddress(&ptr, g_error_word));
    int sms = 0;
    C2KV_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    g_err_ptr[dev] = static_cast<unsigned*>(ptr);
    g_num_sms[dev] = sms;
  }
  if (err) *err = g_err_ptr[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  return C2KV_OK;
}

// SM count for sizing (no GPU needed: falls back to a GB300's 152 SMs).
int sm_count_for_sizing() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
    return sms;
  cudaGetLastError();
  return 152;
}

c2kv_status check_geom(const c2kv_geometry* g) {
  if (g == nullptr) return fail(C2KV_EINVAL, "geometry is null");
  if (g->n_layers < 1 || g->n_q_heads < 1 || g->n_kv_heads < 1)
    return fail(C2KV_EINVAL, "geometry: layer and head counts must be >= 1");
  if (g->n_q_heads % g->n_kv_heads != 0)
    return fail(C2KV_EINVAL, "geometry: n_kv_heads must divide n_q_heads");
  const int grp = g->n_q_heads / g->n_kv_heads;
  if (grp != 1 && grp != 2 && grp != 4 && grp != 5 && grp != 8)
    return fail(C2KV_EINVAL, "geometry: q heads per kv head must be 1, 2, 4, 5 or 8");
  if (g->head_dim != 64 && g->head_dim != 128)
    return fail(C2KV_EINVAL, "geometry: head_dim must be 64 or 128");
  if (!(g->rope_theta > 1.0) || !std::isfinite(g->rope_theta))
    return fail(C2KV_EINVAL, "geometry: rope_theta must be finite and > 1");
  if (g->n_kv_heads * (g->head_dim / 16) > 1024)
    return fail(C2KV_EINVAL, "geometry: too many kv heads");
  return C2KV_OK;
}

void fill_inv_freq(const c2kv_geometry* g, double* out) {
  for (int i = 0; i < g->head_dim / 2; ++i) out[i] = std::pow(g->rope_theta, -2.0 * i / g->head_dim);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Seg {
  size_t k_off, v_off;
  int32_t n_tokens, n_slots, k;
};

}  // namespace

struct c2kv_store_s {
  c2kv_geometry g{};
  int device = 0;
  uint8_t* pool = nullptr;       // pinned host pool
  uint8_t* pool_dev = nullptr;   // the same pool's address on the device (read by the composition kernel)
  size_t pool_bytes = 0, used = 0;
  std::unordered_map<int32_t, Seg> docs;
  cudaStream_t side = nullptr;
  // Events that order the copy stream and the callers' streams, used in
  // turn: an event is recorded again only after kEventRing later records, so
  // that no record waits on an earlier record of the same event still in
  // flight (which held the host thread back to the copies' pace).
  std::vector<cudaEvent_t> ev;
  size_t ev_next = 0;
  std::mutex mu;
  // the last composition into each RoPE table (one per request), which a
  // C2KV_COMPOSE_CONTINUE call must match; at most kMaxTrackedTables tables,
  // the least recently started composition dropped first
  struct Composition {
    std::vector<int32_t> doc_ids, order;
    int32_t k = 0, cap = 0;
    uint32_t flags = 0;
    const void *k_cache = nullptr, *v_cache = nullptr;
    uint64_t seq = 0;   // order in which the compositions started
  };
  std::unordered_map<const void*, Composition> last;
  uint64_t next_seq = 0;
};

namespace {
constexpr int kEventRing = 64;    // events of a store, recorded in turn
constexpr size_t kMaxTrackedTables = 1024;

// Composition plan shared by c2kv_plan and c2kv_compose.
c2kv_status plan_impl(int32_t n_docs, const int32_t* n_tokens, const int32_t* n_slots,
                      const int32_t* order, int32_t* slot_start, int32_t* pos_offset,
                      int32_t* total_slots, int32_t* total_tokens) {
  if (n_docs < 0) return fail(C2KV_EINVAL, "n_docs < 0");
  if (n_docs > 0 && (n_tokens == nullptr || n_slots == nullptr))
    return fail(C2KV_EINVAL, "n_tokens / n_slots is null");
  if (order != nullptr) {
    std::vector<char> seen(n_docs, 0);
    for (int c = 0; c < n_docs; ++c) {
      const int o = order[c];
      if (o < 0 || o >= n_docs || seen[o]) return fail(C2KV_EINVAL, "order is not a permutation of 0..n_docs-1");
      seen[o] = 1;
    }
  }
  int64_t slots = 0, toks = 0;
  for (int c = 0; c < n_docs; ++c) {
    const int d = order ? order[c] : c;
    if (n_tokens[d] < 1) return fail(C2KV_EINVAL, "document with n_tokens < 1");
    if (n_slots[d] < 1 || n_slots[d] > n_tokens[d]) return fail(C2KV_EINVAL, "n_slots must be in [1, n_tokens]");
    if (slot_start) slot_start[c] = (int32_t)slots;
    if (pos_offset) pos_offset[c] = (int32_t)toks;
    slots += n_slots[d];
    toks += n_tokens[d];
    if (slots > INT32_MAX / 2 || toks > INT32_MAX / 2) return fail(C2KV_EINVAL, "composed length overflows int32");
  }
  if (total_slots) *total_slots = (int32_t)slots;
  if (total_tokens) *total_tokens = (int32_t)toks;
  return C2KV_OK;
}

// Scratch of one attention call: split-K partials and arrival counters, and
// for multi-token calls the rotated q in the tensor-core tile layout.
// With tc set (one token per sequence, head_dim 128: the tensor-core decode),
// the partials are two slots per CTA of the launch (one CTA per SM), not
// per split.
struct AttnWs {
  int n_tb, num_splits, split_keys;
  bool tc;
  size_t counters_off, counters_bytes, ml_off, o_off, qrot_off, total;
};

// Bytes of one part (hi or lo) of the rotated-q scratch of the tensor-core
// prefill, 256-byte aligned.
size_t qrot_part_bytes(const c2kv_geometry* g, int batch, int t_len) {
  return align256((size_t)batch * g->n_q_heads * t_len * g->head_dim * 2);
}

// The tensor-core decode serves one token per sequence at head_dim 128, with
// one CTA per SM (at most kDecMaxCtas).
bool use_decode_tc(const c2kv_geometry* g, int t_len) { return t_len == 1 && g->head_dim == 128; }
int decode_tc_ctas(int num_sms) { return std::max(1, std::min(num_sms, kDecMaxCtas)); }

AttnWs attn_workspace(const c2kv_geometry* g, int batch, int t_len, int max_keys, int num_sms) {
  AttnWs w{};
  const int grp = g->n_q_heads / g->n_kv_heads;
  if (use_decode_tc(g, t_len)) {
    w.tc = true;
    w.n_tb = 1;
    w.num_splits = 1;
    w.split_keys = max_keys;
    w.counters_off = 0;
    w.counters_bytes = align256((size_t)kMaxBatch * g->n_kv_heads * sizeof(int32_t));
    size_t off = w.counters_bytes;
    const size_t slots = 2 * (size_t)decode_tc_ctas(num_sms);
    w.ml_off = off;
    off += align256(slots * grp * 2 * sizeof(float));
    w.o_off = off;
    off += align256(slots * grp * g->head_dim * sizeof(float));
    w.qrot_off = off;
    w.total = off;
    return w;
  }
  if (t_len == 1) {
    w.n_tb = 1;
    attn_plan_splits(batch * g->n_kv_heads, max_keys, num_sms, grp, &w.num_splits, &w.split_keys);
  } else {
    // tensor-core prefill: splits are merged inside a cluster (no partials
    // here); the scratch holds only the rotated q
    w.n_tb = prefill_tc_m_tiles(t_len, grp);
    w.num_splits = 1;
    w.split_keys = max_keys;
  }
  const size_t rows = (size_t)batch * t_len * g->n_kv_heads * w.num_splits * grp;
  // The arrival counters sit at the start of every layout, sized for the
  // largest batch, so that no call's other scratch (partials, rotated q)
  // overwrites counters another call relies on being zero.
  size_t off = 0;
  w.counters_off = 0;
  w.counters_bytes = align256((size_t)kMaxBatch * g->n_kv_heads * sizeof(int32_t));
  off += w.counters_bytes;
  if (w.num_splits > 1) {
    w.ml_off = off;
    off += align256(rows * 2 * sizeof(float));
    w.o_off = off;
    off += align256(rows * g->head_dim * sizeof(float));
  }
  w.qrot_off = off;   // rotated q for the tensor-core prefill: bf16 hi part, then lo part
  if (t_len > 1) off += 2 * align256((size_t)batch * g->n_q_heads * t_len * g->head_dim * 2);
  w.total = off;
  return w;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    cudaGetLastError();
  });
  return fn;
}

// bf16 tensor map with a 64-element (128-byte) inner box and 128-byte swizzle.
// rank 2: {d, rows}, box {64, box_rows}; rank 3: {d, keys, blocks} with the
// block stride given, box {64, box_rows, 1}.
c2kv_status encode_map(CUtensorMap* m, const void* base, int rank, uint64_t d, uint64_t n1, uint64_t n2,
                       uint64_t stride2_bytes, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return fail(C2KV_ECUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[3] = {d, n1, n2};
  const cuuint64_t strides[2] = {d * 2, stride2_bytes};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(C2KV_ECUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
  return C2KV_OK;
}

// Multi-token attention on the tensor cores.  kb0/vb0: per-sequence layer-0
// bases of [n_blocks = layers * kv heads][block_rows][d] key/value arrays;
// valid[b] keys of each block are real, the rest read as zeros.
c2kv_status run_prefill_tc(const c2kv_geometry* g, int batch, const void* const* kb0, const void* const* vb0,
                           const int32_t* n_cached, const int32_t* valid, int n_blocks, int block_rows,
                           int layer, int t_len, int max_keys, int mask_mode, int n_doc, int kblk,
                           void* out, const AttnWs& w, uint8_t* ws, cudaStream_t st) {
  unsigned* err = nullptr;
  int sms = 0;
  c2kv_status s = device_state(&err, &sms);
  if (s != C2KV_OK) return s;
  static PrefillTcParams p;   // large (tensor maps); guarded by the mutex below
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&p, 0, sizeof(p));
  const int D = g->head_dim;
  const int grp = g->n_q_heads / g->n_kv_heads;
  p.q_hi = reinterpret_cast<const __nv_bfloat16*>(ws + w.qrot_off);
  p.q_lo = reinterpret_cast<const __nv_bfloat16*>(ws + w.qrot_off + qrot_part_bytes(g, batch, t_len));
  for (int b = 0; b < batch; ++b) {
    const uint64_t stride2 = (uint64_t)block_rows * D * 2;
    s = encode_map(&p.tm_k[b], kb0[b], 3, D, valid[b], n_blocks, stride2, (uint32_t)prefill_tc_key_tile());
    if (s != C2KV_OK) return s;
    s = encode_map(&p.tm_v[b], vb0[b], 3, D, valid[b], n_blocks, stride2, (uint32_t)prefill_tc_key_tile());
    if (s != C2KV_OK) return s;
    p.n_cached[b] = n_cached[b];
  }
  p.out = static_cast<__nv_bfloat16*>(out);
  p.err = err;
  p.batch = batch;
  p.t_len = t_len;
  p.n_q = g->n_q_heads;
  p.n_kv = g->n_kv_heads;
  p.layer = layer;
  const int units = batch * w.n_tb * g->n_kv_heads;
  // every unit's keys are within 2x of each other when each sequence's
  // cached keys are at least its question's
  bool even = mask_mode == kMaskCausal;
  for (int b = 0; b < batch; ++b) even = even && n_cached[b] >= t_len;
  const PrefillTcSchedule sc = prefill_tc_schedule(units, max_keys, sms, D, grp, even);
  p.n_mt = w.n_tb;
  p.mask_mode = mask_mode;
  p.n_doc = n_doc;
  p.kblk = kblk;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  p.unit0 = 0;
  p.n_units = sc.bulk;
  p.num_splits = sc.splits0;
  p.split_keys = sc.keys0;
  C2KV_LAUNCH(launch_prefill_tc(p, D, grp, st));
  if (sc.bulk < units) {
    p.unit0 = sc.bulk;
    p.n_units = units - sc.bulk;
    p.num_splits = sc.splits1;
    p.split_keys = sc.keys1;
    C2KV_LAUNCH(launch_prefill_tc(p, D, grp, st));
  }
  return C2KV_OK;
}

// Test hook: the next n decode launches take their bounded-wait timeout path.
std::atomic<int> g_inject_timeouts{0};

bool take_injected_timeout() {
  int n = g_inject_timeouts.load();
  while (n > 0 && !g_inject_timeouts.compare_exchange_weak(n, n - 1)) {
  }
  return n > 0;
}

// One token per sequence at head_dim 128, on the tensor cores: kb/vb are the
// layer bases [Hkv][cap][d] of each sequence's cache.
c2kv_status run_decode_tc(const c2kv_geometry* g, int batch, const __nv_bfloat16* const* kb,
                          const __nv_bfloat16* const* vb, const CosSin2* const* tabs, const int32_t* n_cached_h,
                          const int32_t* n_cached_d, int cap, int max_keys, const void* q, void* out,
                          void* workspace, size_t workspace_bytes, cudaStream_t st, const void* k_new,
                          const void* v_new, bool overlap) {
  unsigned* err = nullptr;
  int sms = 0;
  c2kv_status s = device_state(&err, &sms);
  if (s != C2KV_OK) return s;
  const AttnWs w = attn_workspace(g, batch, 1, max_keys, sms);
  if (workspace == nullptr || workspace_bytes < w.total)
    return fail(C2KV_EINVAL, "workspace too small: need " + std::to_string(w.total) + " bytes");
  static DecodeTcParams p;   // large (tensor maps); guarded by the mutex below
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&p, 0, sizeof(p));
  const int D = g->head_dim;
  for (int b = 0; b < batch; ++b) {
    const uint64_t stride2 = (uint64_t)cap * D * 2;
    s = encode_map(&p.tm_k[b], kb[b], 3, D, (uint64_t)cap, g->n_kv_heads, stride2, 128);
    if (s != C2KV_OK) return s;
    s = encode_map(&p.tm_v[b], vb[b], 3, D, (uint64_t)cap, g->n_kv_heads, stride2, 128);
    if (s != C2KV_OK) return s;
    p.k_base[b] = const_cast<__nv_bfloat16*>(kb[b]);
    p.v_base[b] = const_cast<__nv_bfloat16*>(vb[b]);
    p.tab[b] = tabs[b];
    p.n_cached_h[b] = n_cached_h ? n_cached_h[b] : 0;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.n_cached_d = n_cached_d;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.part_o = reinterpret_cast<float*>(ws + w.o_off);
  p.part_ml = reinterpret_cast<float*>(ws + w.ml_off);
  p.counters = reinterpret_cast<int32_t*>(ws + w.counters_off);
  p.err = err;
  p.batch = batch;
  p.n_q = g->n_q_heads;
  p.n_kv = g->n_kv_heads;
  p.cap = cap;
  p.max_keys = max_keys;
  p.fuse_append = k_new != nullptr ? 1 : 0;
  p.inject_timeout = take_injected_timeout() ? 1 : 0;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  // Few tiles per SM (short caches, few sequences): the launch is latency-
  // bound and the units' partial merges dominate, so launch one thread-block
  // cluster per unit when that many clusters fit at once; they merge in
  // distributed shared memory.
  const int grp = g->n_q_heads / g->n_kv_heads;
  const int units = batch * g->n_kv_heads;
  const int ctas_max = decode_tc_ctas(sms);
  const int64_t tiles = (int64_t)units * ((max_keys + kDecKeyTile - 1) / kDecKeyTile);
  int ctas = ctas_max;
  if (tiles < (int64_t)kDecClusterTilesPerSm * ctas_max) {
    for (int cs = std::min(16, ctas_max / units); cs >= 2; --cs) {
      if (decode_tc_active_clusters(grp, cs) >= units) {
        p.cluster = cs;
        ctas = units * cs;
        break;
      }
    }
  }
  C2KV_LAUNCH(launch_decode_tc(p, grp, ctas, overlap, st));
  return C2KV_OK;
}

// tabs[b]: per-row cos/sin table of sequence b (token t at row n_cached + t).
c2kv_status run_attention(const c2kv_geometry* g, int batch, const __nv_bfloat16* const* kb,
                          const __nv_bfloat16* const* vb, const CosSin2* const* tabs, const int32_t* n_cached_h,
                          const int32_t* n_cached_d, int cap, int max_keys, int t_len, int mask_mode, int n_doc,
                          int kblk, const void* q, void* out, void* workspace, size_t workspace_bytes,
                          cudaStream_t st, const void* fused_k_new = nullptr, const void* fused_v_new = nullptr,
                          bool overlap = false) {
  if (use_decode_tc(g, t_len))   // any mask is causal for a one-token sequence
    return run_decode_tc(g, batch, kb, vb, tabs, n_cached_h, n_cached_d, cap, max_keys, q, out, workspace,
                         workspace_bytes, st, fused_k_new, fused_v_new, overlap);
  unsigned* err = nullptr;
  int sms = 0;
  c2kv_status s = device_state(&err, &sms);
  if (s != C2KV_OK) return s;
  const AttnWs w = attn_workspace(g, batch, t_len, max_keys, sms);
  if (w.total > 0 && (workspace == nullptr || workspace_bytes < w.total))
    return fail(C2KV_EINVAL, "workspace too small: need " + std::to_string(w.total) + " bytes");
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  for (int b = 0; b < batch; ++b) {
    p.k_base[b] = kb[b];
    p.v_base[b] = vb[b];
    p.tab[b] = tabs[b];
    p.n_cached_h[b] = n_cached_h ? n_cached_h[b] : 0;
  }
  p.n_cached_d = n_cached_d;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = w.num_splits > 1 ? reinterpret_cast<int32_t*>(ws + w.counters_off) : nullptr;
  p.part_ml = w.num_splits > 1 ? reinterpret_cast<float*>(ws + w.ml_off) : nullptr;
  p.part_o = w.num_splits > 1 ? reinterpret_cast<float*>(ws + w.o_off) : nullptr;
  p.err = err;
  p.batch = batch;
  p.t_len = t_len;
  p.n_q = g->n_q_heads;
  p.n_kv = g->n_kv_heads;
  p.cap = cap;
  p.max_keys = max_keys;
  p.num_splits = w.num_splits;
  p.split_keys = w.split_keys;
  p.mask_mode = mask_mode;
  p.n_doc = n_doc;
  p.kblk = kblk;
  // Prefer merging the key splits inside a thread-block cluster (no global
  // partials) when clusters of that many CTAs fit the GPU all at once.
  {
    const int units = batch * g->n_kv_heads;
    int want = sms / units;
    const int by_keys = (max_keys + 63) / 64;
    if (want > by_keys) want = by_keys;
    const int cs = attn_cluster_splits(units, want, g->head_dim, g->n_q_heads / g->n_kv_heads);
    // only when the cluster keeps as many CTAs streaming as the global plan
    if (cs >= 2 && cs >= w.num_splits) {
      int sk = (max_keys + cs - 1) / cs;
      sk = (sk + 7) / 8 * 8;
      const int ns = (max_keys + sk - 1) / sk;
      if (ns >= 2) {
        p.num_splits = ns;
        p.split_keys = sk;
        p.cluster_merge = 1;
      }
    }
  }
  p.inject_timeout = take_injected_timeout() ? 1 : 0;
  p.fuse_append = fused_k_new != nullptr ? 1 : 0;
  p.k_new = static_cast<const __nv_bfloat16*>(fused_k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(fused_v_new);
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)g->head_dim));
  C2KV_LAUNCH(launch_attention(p, g->head_dim, g->n_q_heads / g->n_kv_heads, overlap, st));
  return C2KV_OK;
}

c2kv_status run_append(const c2kv_geometry* g, int batch, __nv_bfloat16* const* kd, __nv_bfloat16* const* vd,
                       const CosSin2* const* tabs, const int32_t* row_h, const int32_t* row_d, int cap, int t_len,
                       const void* k_src, const void* v_src, cudaStream_t st, const void* q_src = nullptr,
                       void* q_dst = nullptr) {
  // q_dst: the rotated-q scratch, bf16 hi part then lo part
  unsigned* err = nullptr;
  c2kv_status s = device_state(&err, nullptr);
  if (s != C2KV_OK) return s;
  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  for (int b = 0; b < batch; ++b) {
    p.k_dst[b] = kd[b];
    p.v_dst[b] = vd[b];
    p.tab[b] = tabs[b];
    p.row_h[b] = row_h ? row_h[b] : 0;
  }
  p.row_d = row_d;
  p.k_src = static_cast<const __nv_bfloat16*>(k_src);
  p.v_src = static_cast<const __nv_bfloat16*>(v_src);
  p.q_src = static_cast<const __nv_bfloat16*>(q_src);
  p.q_dst = static_cast<__nv_bfloat16*>(q_dst);
  p.q_dst_lo = q_dst ? reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(q_dst) + qrot_part_bytes(g, batch, t_len))
                     : nullptr;
  p.err = err;
  p.t_len = t_len;
  p.n_kv = g->n_kv_heads;
  p.n_q = g->n_q_heads;
  p.cap = cap;
  C2KV_LAUNCH(launch_append(p, g->head_dim, batch, st));
  return C2KV_OK;
}

size_t table_bytes(const c2kv_geometry* g, int rows) { return (size_t)rows * (g->head_dim / 2) * sizeof(CosSin2); }

c2kv_status check_caches(int batch, void* const* kc, void* const* vc, int cap) {
  if (batch < 1 || batch > kMaxBatch) return fail(C2KV_EINVAL, "batch must be in [1, 16]");
  if (kc == nullptr || vc == nullptr) return fail(C2KV_EINVAL, "cache pointer arrays are null");
  if (cap < 1) return fail(C2KV_EINVAL, "cap must be >= 1");
  for (int b = 0; b < batch; ++b) {
    if (kc[b] == nullptr || vc[b] == nullptr) return fail(C2KV_EINVAL, "a cache pointer is null");
    if ((reinterpret_cast<uintptr_t>(kc[b]) | reinterpret_cast<uintptr_t>(vc[b])) & 15)
      return fail(C2KV_EINVAL, "cache pointers must be 16-byte aligned");
  }
  return C2KV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" {

const char* c2kv_last_error(void) { return g_err.c_str(); }

const char* c2kv_version(void) { return "c2kv-gb300 0.1 (sm_103a)"; }

c2kv_status c2kv_store_create(const c2kv_geometry* geom, size_t pinned_bytes, c2kv_store* out) {
  c2kv_status s = check_geom(geom);
  if (s != C2KV_OK) return s;
  if (out == nullptr) return fail(C2KV_EINVAL, "out is null");
  *out = nullptr;
  c2kv_store st = new (std::nothrow) c2kv_store_s();
  if (st == nullptr) return fail(C2KV_ENOMEM, "host allocation failed");
  st->g = *geom;
  cudaError_t e = cudaGetDevice(&st->device);
  if (e == cudaSuccess && pinned_bytes > 0) {
    e = cudaHostAlloc(reinterpret_cast<void**>(&st->pool), pinned_bytes, cudaHostAllocMapped);
    if (e == cudaSuccess) {
      e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&st->pool_dev), st->pool, 0);
      if (e != cudaSuccess) {
        cudaFreeHost(st->pool);
        st->pool = nullptr;
      }
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      delete st;
      return fail(C2KV_ENOMEM, std::string("cudaHostAlloc of the pinned pool failed: ") + cudaGetErrorString(e));
    }
    st->pool_bytes = pinned_bytes;
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st->side, cudaStreamNonBlocking);
  for (int i = 0; e == cudaSuccess && i < kEventRing; ++i) {
    cudaEvent_t ev;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) st->ev.push_back(ev);
  }
  if (e != cudaSuccess) {
    c2kv_store_destroy(st);
    return fail(C2KV_ECUDA, std::string("store setup failed: ") + cudaGetErrorString(e));
  }
  *out = st;
  return C2KV_OK;
}

void c2kv_store_destroy(c2kv_store st) {
  if (st == nullptr) return;
  if (st->side) {
    cudaStreamSynchronize(st->side);
    cudaStreamDestroy(st->side);
  }
  for (cudaEvent_t ev : st->ev) cudaEventDestroy(ev);
  if (st->pool) cudaFreeHost(st->pool);
  delete st;
}

c2kv_status c2kv_store_segments(c2kv_store st, int32_t n_docs, const int32_t* doc_ids,
                                const int32_t* n_tokens, const int32_t* n_slots, int32_t k,
                                const void* const* k_pre, const void* const* v) {
  if (st == nullptr) return fail(C2KV_EINVAL, "store is null");
  if (n_docs < 0) return fail(C2KV_EINVAL, "n_docs < 0");
  if (n_docs == 0) return C2KV_OK;
  if (!doc_ids || !n_tokens || !n_slots || !k_pre || !v) return fail(C2KV_EINVAL, "null argument");
  if (k < 1) return fail(C2KV_EINVAL, "k must be >= 1");
  std::lock_guard<std::mutex> lk(st->mu);
  const c2kv_geometry& g = st->g;
  const size_t row = (size_t)g.n_layers * g.n_kv_heads * g.head_dim * 2;   // bytes per slot (K or V)
  size_t need = 0;
  std::unordered_set<int32_t> ids;
  for (int i = 0; i < n_docs; ++i) {
    if (n_tokens[i] < 1) return fail(C2KV_EINVAL, "n_tokens must be >= 1");
    if (n_slots[i] < 1 || n_slots[i] > n_tokens[i]) return fail(C2KV_EINVAL, "n_slots must be in [1, n_tokens]");
    if (!k_pre[i] || !v[i]) return fail(C2KV_EINVAL, "segment pointer is null");
    if (st->docs.count(doc_ids[i]) || !ids.insert(doc_ids[i]).second)
      return fail(C2KV_EINVAL, "document id " + std::to_string(doc_ids[i]) + " is already stored");
    need += 2 * align256(row * n_slots[i]);
  }
  if (st->used + need > st->pool_bytes)
    return fail(C2KV_ENOMEM, "pinned pool full: need " + std::to_string(need) + " more bytes");
  for (int i = 0; i < n_docs; ++i) {
    const size_t bytes = row * n_slots[i];
    Seg sg;
    sg.k_off = st->used;
    std::memcpy(st->pool + sg.k_off, k_pre[i], bytes);
    st->used += align256(bytes);
    sg.v_off = st->used;
    std::memcpy(st->pool + sg.v_off, v[i], bytes);
    st->used += align256(bytes);
    sg.n_tokens = n_tokens[i];
    sg.n_slots = n_slots[i];
    sg.k = k;
    st->docs[doc_ids[i]] = sg;
  }
  return C2KV_OK;
}

namespace {
// Store file: a header, then per document (ascending ids) its record, its K
// rows and its V rows exactly as held in the pool ([layer][kv head][slot][d]
// bf16), all in host byte order.
constexpr char kStoreMagic[8] = {'C', '2', 'K', 'V', 'S', 'T', 'O', 'R'};
constexpr uint32_t kStoreVersion = 1;
struct StoreFileHeader {
  char magic[8];
  uint32_t version, reserved;
  int32_t n_layers, n_q_heads, n_kv_heads, head_dim;
  double rope_theta;
  uint64_t n_docs;
};
struct StoreFileDoc {
  int32_t doc_id, n_tokens, n_slots, k;
};
}  // namespace

c2kv_status c2kv_store_save(c2kv_store st, const char* path) {
  if (st == nullptr || path == nullptr) return fail(C2KV_EINVAL, "store or path is null");
  std::lock_guard<std::mutex> lk(st->mu);
  const c2kv_geometry& g = st->g;
  const size_t row = (size_t)g.n_layers * g.n_kv_heads * g.head_dim * 2;
  std::vector<int32_t> ids;
  for (const auto& kv : st->docs) ids.push_back(kv.first);
  std::sort(ids.begin(), ids.end());
  FILE* f = std::fopen(path, "wb");
  if (f == nullptr) return fail(C2KV_EIO, std::string("cannot open ") + path + " for writing");
  StoreFileHeader hd;
  std::memset(&hd, 0, sizeof(hd));
  std::memcpy(hd.magic, kStoreMagic, sizeof(kStoreMagic));
  hd.version = kStoreVersion;
  hd.n_layers = g.n_layers;
  hd.n_q_heads = g.n_q_heads;
  hd.n_kv_heads = g.n_kv_heads;
  hd.head_dim = g.head_dim;
  hd.rope_theta = g.rope_theta;
  hd.n_docs = ids.size();
  bool ok = std::fwrite(&hd, sizeof(hd), 1, f) == 1;
  for (size_t i = 0; ok && i < ids.size(); ++i) {
    const Seg& sg = st->docs.at(ids[i]);
    const StoreFileDoc rec{ids[i], sg.n_tokens, sg.n_slots, sg.k};
    const size_t bytes = row * sg.n_slots;
    ok = std::fwrite(&rec, sizeof(rec), 1, f) == 1 && std::fwrite(st->pool + sg.k_off, 1, bytes, f) == bytes &&
         std::fwrite(st->pool + sg.v_off, 1, bytes, f) == bytes;
  }
  if (std::fclose(f) != 0) ok = false;
  if (!ok) return fail(C2KV_EIO, std::string("writing ") + path + " failed");
  return C2KV_OK;
}

c2kv_status c2kv_store_load(c2kv_store st, const char* path) {
  if (st == nullptr || path == nullptr) return fail(C2KV_EINVAL, "store or path is null");
  FILE* f = std::fopen(path, "rb");
  if (f == nullptr) return fail(C2KV_EIO, std::string("cannot open ") + path);
  struct Closer {
    FILE* f;
    ~Closer() { std::fclose(f); }
  } closer{f};
  StoreFileHeader hd;
  if (std::fread(&hd, sizeof(hd), 1, f) != 1) return fail(C2KV_EIO, std::string(path) + ": truncated header");
  if (std::memcmp(hd.magic, kStoreMagic, sizeof(kStoreMagic)) != 0 || hd.version != kStoreVersion)
    return fail(C2KV_EINVAL, std::string(path) + " is not a c2kv store file of version 1");
  const c2kv_geometry& g = st->g;
  if (hd.n_layers != g.n_layers || hd.n_q_heads != g.n_q_heads || hd.n_kv_heads != g.n_kv_heads ||
      hd.head_dim != g.head_dim || hd.rope_theta != g.rope_theta)
    return fail(C2KV_EINVAL, std::string(path) + " was saved with another geometry");
  const size_t row = (size_t)g.n_layers * g.n_kv_heads * g.head_dim * 2;
  std::vector<uint8_t> kb, vb;
  for (uint64_t i = 0; i < hd.n_docs; ++i) {
    StoreFileDoc rec;
    if (std::fread(&rec, sizeof(rec), 1, f) != 1) return fail(C2KV_EIO, std::string(path) + ": truncated");
    if (rec.n_tokens < 1 || rec.n_slots < 1 || rec.n_slots > rec.n_tokens || rec.k < 1)
      return fail(C2KV_EINVAL, std::string(path) + ": bad document record");
    const size_t bytes = row * (size_t)rec.n_slots;
    {
      std::lock_guard<std::mutex> lk(st->mu);
      if (st->used + 2 * align256(bytes) > st->pool_bytes)
        return fail(C2KV_ENOMEM, "pinned pool full: document " + std::to_string(rec.doc_id) + " does not fit");
    }
    kb.resize(bytes);
    vb.resize(bytes);
    if (std::fread(kb.data(), 1, bytes, f) != bytes || std::fread(vb.data(), 1, bytes, f) != bytes)
      return fail(C2KV_EIO, std::string(path) + ": truncated");
    const void* kp = kb.data();
    const void* vp = vb.data();
    const c2kv_status s = c2kv_store_segments(st, 1, &rec.doc_id, &rec.n_tokens, &rec.n_slots, rec.k, &kp, &vp);
    if (s != C2KV_OK) return s;
  }
  return C2KV_OK;
}

c2kv_status c2kv_store_lookup(c2kv_store st, int32_t doc_id, int32_t* n_tokens, int32_t* n_slots, int32_t* k) {
  if (st == nullptr) return fail(C2KV_EINVAL, "store is null");
  std::lock_guard<std::mutex> lk(st->mu);
  auto it = st->docs.find(doc_id);
  if (it == st->docs.end()) return fail(C2KV_ENOTFOUND, "unknown document id " + std::to_string(doc_id));
  if (n_tokens) *n_tokens = it->second.n_tokens;
  if (n_slots) *n_slots = it->second.n_slots;
  if (k) *k = it->second.k;
  return C2KV_OK;
}

c2kv_status c2kv_plan(int32_t n_docs, const int32_t* n_tokens, const int32_t* n_slots, const int32_t* order,
                      int32_t* slot_start, int32_t* pos_offset, int32_t* total_slots, int32_t* total_tokens) {
  return plan_impl(n_docs, n_tokens, n_slots, order, slot_start, pos_offset, total_slots, total_tokens);
}

c2kv_status c2kv_compose(c2kv_store st, int32_t n_docs, const int32_t* doc_ids, const int32_t* order, int32_t k,
                         void* k_cache, void* v_cache, int32_t cap, void* rope_table_out, int32_t* pos_dev_out,
                         int32_t* n_slots_out, int32_t* next_pos_out, void* stream) {
  if (st == nullptr) return fail(C2KV_EINVAL, "store is null");
  return c2kv_compose_layers(st, n_docs, doc_ids, order, k, 0u, 0, st->g.n_layers, k_cache, v_cache, cap,
                             rope_table_out, pos_dev_out, n_slots_out, next_pos_out, stream);
}

c2kv_status c2kv_compose_layers(c2kv_store st, int32_t n_docs, const int32_t* doc_ids, const int32_t* order,
                                int32_t k, uint32_t flags, int32_t layer_begin, int32_t layer_end, void* k_cache,
                                void* v_cache, int32_t cap, void* rope_table_out, int32_t* pos_dev_out,
                                int32_t* n_slots_out, int32_t* next_pos_out, void* stream) {
  if (st == nullptr) return fail(C2KV_EINVAL, "store is null");
  if (flags & ~(C2KV_COMPOSE_NO_REALIGN | C2KV_COMPOSE_CONTINUE)) return fail(C2KV_EINVAL, "unknown flags");
  if (layer_begin < 0 || layer_end > st->g.n_layers || layer_begin >= layer_end)
    return fail(C2KV_EINVAL, "need 0 <= layer_begin < layer_end <= n_layers");
  const bool cont = (flags & C2KV_COMPOSE_CONTINUE) != 0;
  const bool realign = (flags & C2KV_COMPOSE_NO_REALIGN) == 0;
  if (n_docs < 0 || n_docs > kMaxDocsPerCompose)
    return fail(C2KV_EINVAL, "n_docs must be in [0, " + std::to_string(kMaxDocsPerCompose) + "]");
  if (n_docs > 0 && doc_ids == nullptr) return fail(C2KV_EINVAL, "doc_ids is null");
  if (k < 1) return fail(C2KV_EINVAL, "k must be >= 1");
  if (cap < 0) return fail(C2KV_EINVAL, "cap < 0");
  std::lock_guard<std::mutex> lk(st->mu);
  const c2kv_geometry& g = st->g;
  std::vector<Seg> segs(n_docs);
  std::vector<int32_t> ntok(n_docs), nsl(n_docs);
  for (int i = 0; i < n_docs; ++i) {
    auto it = st->docs.find(doc_ids[i]);
    if (it == st->docs.end()) return fail(C2KV_ENOTFOUND, "unknown document id " + std::to_string(doc_ids[i]));
    if (it->second.k != k)
      return fail(C2KV_EINVAL, "document " + std::to_string(doc_ids[i]) + " was stored with k=" +
                                   std::to_string(it->second.k));
    segs[i] = it->second;
    ntok[i] = segs[i].n_tokens;
    nsl[i] = segs[i].n_slots;
  }
  std::vector<int32_t> slot0(n_docs), off(n_docs);
  int32_t total = 0, l_tot = 0;
  c2kv_status s = plan_impl(n_docs, ntok.data(), nsl.data(), order, slot0.data(), off.data(), &total, &l_tot);
  if (s != C2KV_OK) return s;
  if (total > cap)
    return fail(C2KV_ECAPACITY, "composed slots " + std::to_string(total) + " exceed cap " + std::to_string(cap));
  if ((int64_t)l_tot + (cap - total) > INT32_MAX / 2) return fail(C2KV_EINVAL, "positions overflow int32");
  const uint32_t base_flags = flags & ~C2KV_COMPOSE_CONTINUE;
  if (cont) {
    const auto it = st->last.find(rope_table_out);
    const std::vector<int32_t> ids(doc_ids, doc_ids + n_docs);
    const std::vector<int32_t> ord = order ? std::vector<int32_t>(order, order + n_docs) : std::vector<int32_t>();
    if (it == st->last.end() || it->second.doc_ids != ids || it->second.order != ord || it->second.k != k ||
        it->second.cap != cap || it->second.flags != base_flags || it->second.k_cache != k_cache ||
        it->second.v_cache != v_cache)
      return fail(C2KV_EINVAL, "C2KV_COMPOSE_CONTINUE does not follow a composition of the same request");
  }
  if (n_slots_out) *n_slots_out = total;
  if (next_pos_out) *next_pos_out = l_tot;
  if (cap == 0) return C2KV_OK;
  if (rope_table_out == nullptr) return fail(C2KV_EINVAL, "rope_table_out is null");
  if (total > 0 && (k_cache == nullptr || v_cache == nullptr)) return fail(C2KV_EINVAL, "cache pointer is null");
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(rope_table_out))
    return fail(C2KV_EINVAL, "cache and table pointers must be 16-byte aligned");
  int dev = -1;
  C2KV_CUDA(cudaGetDevice(&dev));
  if (dev != st->device) return fail(C2KV_EINVAL, "current device differs from the store's device");
  s = device_state(nullptr, nullptr);
  if (s != C2KV_OK) return s;

  cudaStream_t us = static_cast<cudaStream_t>(stream);
  const int D = g.head_dim, H = g.n_kv_heads;
  CosSin2* tab = static_cast<CosSin2*>(rope_table_out);

  // The cos/sin table of every cache row is built on the caller's stream by
  // the first call of a composition.
  static TableParams tp;   // large (segment table); guarded by the store mutex and g_tab_mu
  static std::mutex g_tab_mu;
  if (!cont) {
    st->last.erase(rope_table_out);
    std::lock_guard<std::mutex> tl(g_tab_mu);
    std::memset(&tp, 0, sizeof(tp));
    tp.tab = tab;
    tp.pos_out = pos_dev_out;
    tp.rows = cap;
    tp.half = D / 2;
    tp.mode = kTableComposed;
    tp.n_total = total;
    tp.l_tot = l_tot;
    tp.k = k;
    tp.n_docs = n_docs;
    fill_inv_freq(&g, tp.inv_freq);
    for (int c = 0; c < n_docs; ++c) {
      const int d = order ? order[c] : c;
      tp.seg[c].slot0 = slot0[c];
      tp.seg[c].n_slots = nsl[d];
      tp.seg[c].off = realign ? off[c] : 0;   // no re-alignment: extraction positions
      tp.seg[c].n_tokens = ntok[d];
    }
    C2KV_LAUNCH(launch_rope_table(tp, us));
    if (st->last.size() >= kMaxTrackedTables) {   // this table's entry was erased above
      auto oldest = st->last.begin();
      for (auto it = st->last.begin(); it != st->last.end(); ++it)
        if (it->second.seq < oldest->second.seq) oldest = it;
      st->last.erase(oldest);
    }
    auto& lc = st->last[rope_table_out];
    lc.seq = st->next_seq++;
    lc.doc_ids.assign(doc_ids, doc_ids + n_docs);
    if (order)
      lc.order.assign(order, order + n_docs);
    else
      lc.order.clear();
    lc.k = k;
    lc.cap = cap;
    lc.flags = base_flags;
    lc.k_cache = k_cache;
    lc.v_cache = v_cache;
  }
  if (total == 0) return C2KV_OK;

  // The composition kernel runs on the store's stream, after the caller's
  // earlier work and the table (a continuation: after the kernel of the call
  // it continues), so that work the caller enqueues between calls (the
  // question prefill of the layers already composed) overlaps it; the
  // caller's stream waits for it.
  if (!cont) {
    const cudaEvent_t fork = st->ev[st->ev_next++ % st->ev.size()];
    C2KV_CUDA(cudaEventRecord(fork, us));
    C2KV_CUDA(cudaStreamWaitEvent(st->side, fork, 0));
  }
  static ComposeParams cp;   // large (segment table); guarded by the store mutex and g_cmp_mu
  static std::mutex g_cmp_mu;
  {
    std::lock_guard<std::mutex> cl(g_cmp_mu);
    std::memset(&cp, 0, sizeof(cp));
    cp.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    cp.v_cache = static_cast<__nv_bfloat16*>(v_cache);
    cp.tab = tab;
    cp.cap = cap;
    cp.n_kv = H;
    cp.layer0 = layer_begin;
    cp.layer1 = layer_end;
    cp.n_total = total;
    cp.n_docs = n_docs;
    for (int c = 0; c < n_docs; ++c) {
      const Seg& sg = segs[order ? order[c] : c];
      cp.seg[c].k = reinterpret_cast<const __nv_bfloat16*>(st->pool_dev + sg.k_off);
      cp.seg[c].v = reinterpret_cast<const __nv_bfloat16*>(st->pool_dev + sg.v_off);
      cp.seg[c].slot0 = slot0[c];
      cp.seg[c].n_slots = sg.n_slots;
    }
    C2KV_LAUNCH(launch_compose(cp, D, st->side));
  }
  const cudaEvent_t landed = st->ev[st->ev_next++ % st->ev.size()];
  C2KV_CUDA(cudaEventRecord(landed, st->side));
  C2KV_CUDA(cudaStreamWaitEvent(us, landed, 0));
  return C2KV_OK;
}

size_t c2kv_rope_table_bytes(const c2kv_geometry* geom, int32_t rows) {
  if (check_geom(geom) != C2KV_OK || rows < 0) return 0;
  return table_bytes(geom, rows);
}

c2kv_status c2kv_rope_table(const c2kv_geometry* geom, const int32_t* pos_dev, int32_t rows, void* table_out,
                            void* stream) {
  c2kv_status s = check_geom(geom);
  if (s != C2KV_OK) return s;
  if (rows < 0) return fail(C2KV_EINVAL, "rows < 0");
  if (rows == 0) return C2KV_OK;
  if (pos_dev == nullptr || table_out == nullptr) return fail(C2KV_EINVAL, "null pointer");
  if (!aligned16(table_out)) return fail(C2KV_EINVAL, "table_out must be 16-byte aligned");
  s = device_state(nullptr, nullptr);
  if (s != C2KV_OK) return s;
  TableParams p;
  std::memset(&p, 0, sizeof(p));
  p.tab = static_cast<CosSin2*>(table_out);
  p.pos_in = pos_dev;
  p.rows = rows;
  p.half = geom->head_dim / 2;
  p.mode = kTableExplicit;
  fill_inv_freq(geom, p.inv_freq);
  C2KV_LAUNCH(launch_rope_table(p, static_cast<cudaStream_t>(stream)));
  return C2KV_OK;
}

size_t c2kv_attend_workspace_size(const c2kv_geometry* geom, int32_t batch, int32_t t_len, int32_t max_keys) {
  if (check_geom(geom) != C2KV_OK || batch < 1 || t_len < 1 || max_keys < 1) return 0;
  const AttnWs w = attn_workspace(geom, batch, t_len, max_keys, sm_count_for_sizing());
  return std::max<size_t>(w.total, 256);
}

size_t c2kv_masked_extra_bytes(const c2kv_geometry* geom, int32_t n_tokens) {
  if (check_geom(geom) != C2KV_OK || n_tokens < 1) return 0;
  return 2 * align256((size_t)geom->n_kv_heads * n_tokens * geom->head_dim * 2) + align256(table_bytes(geom, n_tokens));
}

c2kv_status c2kv_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (bytes == 0) return C2KV_OK;
  if (workspace == nullptr) return fail(C2KV_EINVAL, "workspace is null");
  C2KV_CUDA(cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)));
  return C2KV_OK;
}

c2kv_status c2kv_attend_prefill(const c2kv_geometry* geom, int32_t layer, int32_t batch, void* const* k_caches,
                                void* const* v_caches, const void* const* rope_tables, int32_t cap,
                                const int32_t* n_cached, int32_t q_len, const void* q, const void* k_new,
                                const void* v_new, void* out, void* workspace, size_t workspace_bytes,
                                void* stream) {
  c2kv_status s = check_geom(geom);
  if (s != C2KV_OK) return s;
  if (layer < 0 || layer >= geom->n_layers) return fail(C2KV_EINVAL, "layer out of range");
  s = check_caches(batch, k_caches, v_caches, cap);
  if (s != C2KV_OK) return s;
  if (q_len < 1) return fail(C2KV_EINVAL, "q_len must be >= 1");
  if (!n_cached || !rope_tables) return fail(C2KV_EINVAL, "n_cached / rope_tables is null");
  if (!q || !k_new || !v_new || !out) return fail(C2KV_EINVAL, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new))
    return fail(C2KV_EINVAL, "q / k_new / v_new must be 16-byte aligned");
  int max_keys = 0;
  const CosSin2* tabs[kMaxBatch];
  for (int b = 0; b < batch; ++b) {
    if (n_cached[b] < 0) return fail(C2KV_EINVAL, "negative n_cached");
    if ((int64_t)n_cached[b] + q_len > cap)
      return fail(C2KV_ECAPACITY, "n_cached + q_len exceeds cap for sequence " + std::to_string(b));
    if (rope_tables[b] == nullptr || !aligned16(rope_tables[b])) return fail(C2KV_EINVAL, "bad rope table pointer");
    tabs[b] = static_cast<const CosSin2*>(rope_tables[b]);
    max_keys = std::max(max_keys, n_cached[b] + q_len);
  }
  const size_t lstride = (size_t)geom->n_kv_heads * cap * geom->head_dim;
  __nv_bfloat16* kb[kMaxBatch];
  __nv_bfloat16* vb[kMaxBatch];
  for (int b = 0; b < batch; ++b) {
    kb[b] = static_cast<__nv_bfloat16*>(k_caches[b]) + layer * lstride;
    vb[b] = static_cast<__nv_bfloat16*>(v_caches[b]) + layer * lstride;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (q_len == 1) {
    s = run_append(geom, batch, kb, vb, tabs, n_cached, nullptr, cap, 1, k_new, v_new, st);
    if (s != C2KV_OK) return s;
    return run_attention(geom, batch, kb, vb, tabs, n_cached, nullptr, cap, max_keys, 1, kMaskCausal, 0, 0, q, out,
                         workspace, workspace_bytes, st);
  }
  int sms = 0;
  s = device_state(nullptr, &sms);
  if (s != C2KV_OK) return s;
  const AttnWs w = attn_workspace(geom, batch, q_len, max_keys, sms);
  if (workspace == nullptr || workspace_bytes < w.total)
    return fail(C2KV_EINVAL, "workspace too small: need " + std::to_string(w.total) + " bytes");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  s = run_append(geom, batch, kb, vb, tabs, n_cached, nullptr, cap, q_len, k_new, v_new, st, q, ws + w.qrot_off);
  if (s != C2KV_OK) return s;
  const void* k0[kMaxBatch];
  const void* v0[kMaxBatch];
  int32_t valid[kMaxBatch];
  for (int b = 0; b < batch; ++b) {
    k0[b] = k_caches[b];
    v0[b] = v_caches[b];
    valid[b] = n_cached[b] + q_len;
  }
  return run_prefill_tc(geom, batch, k0, v0, n_cached, valid, geom->n_layers * geom->n_kv_heads, cap, layer,
                        q_len, max_keys, kMaskCausal, 0, 0, out, w, ws, st);
}

c2kv_status c2kv_attend_decode(const c2kv_geometry* geom, int32_t layer, int32_t batch, void* const* k_caches,
                               void* const* v_caches, const void* const* rope_tables, int32_t cap,
                               const int32_t* n_cached_dev, int32_t max_keys, const void* q, const void* k_new,
                               const void* v_new, void* out, void* workspace, size_t workspace_bytes,
                               uint32_t flags, void* stream) {
  c2kv_status s = check_geom(geom);
  if (flags & ~uint32_t(C2KV_DECODE_OVERLAP_PREVIOUS)) return fail(C2KV_EINVAL, "unknown decode flags");
  if (s != C2KV_OK) return s;
  if (layer < 0 || layer >= geom->n_layers) return fail(C2KV_EINVAL, "layer out of range");
  s = check_caches(batch, k_caches, v_caches, cap);
  if (s != C2KV_OK) return s;
  if (!n_cached_dev || !rope_tables) return fail(C2KV_EINVAL, "n_cached_dev / rope_tables is null");
  if (max_keys < 1 || max_keys > cap) return fail(C2KV_EINVAL, "max_keys must be in [1, cap]");
  if (!q || !k_new || !v_new || !out) return fail(C2KV_EINVAL, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new))
    return fail(C2KV_EINVAL, "q / k_new / v_new must be 16-byte aligned");
  const size_t lstride = (size_t)geom->n_kv_heads * cap * geom->head_dim;
  __nv_bfloat16* kb[kMaxBatch];
  __nv_bfloat16* vb[kMaxBatch];
  const CosSin2* tabs[kMaxBatch];
  for (int b = 0; b < batch; ++b) {
    if (rope_tables[b] == nullptr || !aligned16(rope_tables[b])) return fail(C2KV_EINVAL, "bad rope table pointer");
    tabs[b] = static_cast<const CosSin2*>(rope_tables[b]);
    kb[b] = static_cast<__nv_bfloat16*>(k_caches[b]) + layer * lstride;
    vb[b] = static_cast<__nv_bfloat16*>(v_caches[b]) + layer * lstride;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // One launch: the kernel rotates and stores the new key/value itself.
  return run_attention(geom, batch, kb, vb, tabs, nullptr, n_cached_dev, cap, max_keys, 1, kMaskCausal, 0, 0, q, out,
                       workspace, workspace_bytes, st, k_new, v_new, (flags & C2KV_DECODE_OVERLAP_PREVIOUS) != 0);
}

c2kv_status c2kv_seq_advance(int32_t batch, int32_t* n_cached_dev, int32_t delta, void* stream) {
  if (batch < 1 || batch > 32) return fail(C2KV_EINVAL, "batch must be in [1, 32]");
  if (!n_cached_dev) return fail(C2KV_EINVAL, "null device array");
  C2KV_LAUNCH(launch_advance(batch, n_cached_dev, delta, static_cast<cudaStream_t>(stream)));
  return C2KV_OK;
}

c2kv_status c2kv_attend_masked(const c2kv_geometry* geom, int32_t mask, int32_t n_doc, int32_t n_slot, int32_t k,
                               const void* q, const void* kk, const void* v, void* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  c2kv_status s = check_geom(geom);
  if (s != C2KV_OK) return s;
  if (mask != C2KV_MASK_CAUSAL && mask != C2KV_MASK_STRUCTURED && mask != C2KV_MASK_ANCHOR)
    return fail(C2KV_EINVAL, "unknown mask");
  if (n_doc < 1 || n_slot < 0) return fail(C2KV_EINVAL, "need n_doc >= 1 and n_slot >= 0");
  if (mask == C2KV_MASK_CAUSAL && n_slot != 0) return fail(C2KV_EINVAL, "causal mask takes n_slot = 0");
  if (mask != C2KV_MASK_CAUSAL && k < 1) return fail(C2KV_EINVAL, "k must be >= 1");
  if ((int64_t)n_doc + n_slot > (1 << 24)) return fail(C2KV_EINVAL, "sequence too long");
  if (!q || !kk || !v || !out || !workspace) return fail(C2KV_EINVAL, "null pointer");
  if (!aligned16(q) || !aligned16(kk) || !aligned16(v) || !aligned16(workspace))
    return fail(C2KV_EINVAL, "pointers must be 16-byte aligned");
  const int N = n_doc + n_slot;
  const size_t attn_bytes = c2kv_attend_workspace_size(geom, 1, N, N);
  const size_t extra = c2kv_masked_extra_bytes(geom, N);
  if (workspace_bytes < align256(attn_bytes) + extra)
    return fail(C2KV_EINVAL, "workspace too small: need " + std::to_string(align256(attn_bytes) + extra));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t kv_bytes = align256((size_t)geom->n_kv_heads * N * geom->head_dim * 2);
  __nv_bfloat16* krot = reinterpret_cast<__nv_bfloat16*>(ws + align256(attn_bytes));
  __nv_bfloat16* vt = reinterpret_cast<__nv_bfloat16*>(ws + align256(attn_bytes) + kv_bytes);
  CosSin2* tab = reinterpret_cast<CosSin2*>(ws + align256(attn_bytes) + 2 * kv_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = device_state(nullptr, nullptr);
  if (s != C2KV_OK) return s;
  // Rows are the sequence's tokens: extraction positions (documents at
  // 0..n_doc-1, slot or anchor s at min((s+1)k, n_doc) - 1), or t for the
  // causal mask.
  const bool causal = mask == C2KV_MASK_CAUSAL;
  const int kblk = causal ? 1 : k;
  TableParams tp;
  std::memset(&tp, 0, sizeof(tp));
  tp.tab = tab;
  tp.rows = N;
  tp.half = geom->head_dim / 2;
  tp.mode = kTableExtraction;
  tp.n_doc = causal ? N : n_doc;
  tp.kblk = kblk;
  fill_inv_freq(geom, tp.inv_freq);
  C2KV_LAUNCH(launch_rope_table(tp, st));
  const int32_t zero = 0;
  const CosSin2* tabs[1] = {tab};
  const int mmode = mask == C2KV_MASK_STRUCTURED ? kMaskStructured : mask == C2KV_MASK_ANCHOR ? kMaskAnchor
                                                                                            : kMaskCausal;
  if (N == 1) {   // one document token and no slot or anchor
    s = run_append(geom, 1, &krot, &vt, tabs, &zero, nullptr, N, N, kk, v, st);
    if (s != C2KV_OK) return s;
    const __nv_bfloat16* kb = krot;
    const __nv_bfloat16* vb = vt;
    return run_attention(geom, 1, &kb, &vb, tabs, &zero, nullptr, N, N, N,
                         mmode == kMaskAnchor ? kMaskCausal : mmode, n_doc, kblk, q, out, workspace, attn_bytes, st);
  }
  int sms = 0;
  s = device_state(nullptr, &sms);
  if (s != C2KV_OK) return s;
  const AttnWs w = attn_workspace(geom, 1, N, N, sms);
  s = run_append(geom, 1, &krot, &vt, tabs, &zero, nullptr, N, N, kk, v, st, q, ws + w.qrot_off);
  if (s != C2KV_OK) return s;
  const void* k0 = krot;
  const void* v0 = vt;
  return run_prefill_tc(geom, 1, &k0, &v0, &zero, &N, geom->n_kv_heads, N, 0, N, N, mmode, n_doc, kblk, out, w,
                        ws, st);
}

// Linear workspace: the per-tile arrival counters in a fixed region at offset
// 0 (sized for the largest tile count, so that calls with other shapes that
// share the workspace never write their partials over counters another call
// relies on being zero), then two partial tiles per CTA.
constexpr int kLinearMaxTiles = 8192;
constexpr size_t kLinearCountersBytes = (size_t)kLinearMaxTiles * sizeof(int32_t);

// The linear kernel runs two CTAs per SM: each keeps ~100 KB of weight tiles
// in flight, and streaming an SM's share of HBM at the loaded latency takes
// about twice that.
int linear_ctas(int num_sms) { return std::min(2 * std::max(1, num_sms), 512); }

size_t c2kv_linear_workspace_size(int32_t tokens, int32_t n_out) {
  if (tokens < 1 || tokens > 256 || n_out < 128 || n_out % 128 != 0 || n_out / 128 > kLinearMaxTiles) return 0;
  const int n_pad = (tokens + 15) / 16 * 16;
  const size_t ctas = (size_t)linear_ctas(sm_count_for_sizing());
  return kLinearCountersBytes + 2 * ctas * n_pad * 128 * sizeof(float);
}

c2kv_status c2kv_linear(const void* x, int32_t tokens, int32_t k_in, const void* w, int32_t n_out, int32_t epilogue,
                        const void* residual, void* y, void* y2, void* y3, int32_t split1, int32_t split2,
                        void* workspace, size_t workspace_bytes, uint32_t flags, void* stream) {
  if (flags & ~uint32_t(C2KV_LINEAR_OVERLAP_PREVIOUS)) return fail(C2KV_EINVAL, "unknown linear flags");
  if (tokens < 1 || tokens > 256) return fail(C2KV_EINVAL, "tokens must be in [1, 256]");
  if (k_in < 64 || k_in % 64 != 0) return fail(C2KV_EINVAL, "k_in must be a positive multiple of 64");
  if (n_out < 128 || n_out % 128 != 0 || n_out / 128 > kLinearMaxTiles)
    return fail(C2KV_EINVAL, "n_out must be a positive multiple of 128, at most 1048576");
  if (epilogue < C2KV_LINEAR_STORE || epilogue > C2KV_LINEAR_SWIGLU) return fail(C2KV_EINVAL, "unknown epilogue");
  if (!x || !w || !y || !workspace) return fail(C2KV_EINVAL, "null pointer");
  if (epilogue == C2KV_LINEAR_ADD && !residual) return fail(C2KV_EINVAL, "residual is null");
  if (epilogue == C2KV_LINEAR_SPLIT3) {
    if (!y2 || !y3) return fail(C2KV_EINVAL, "y2 / y3 is null");
    if (!(0 < split1 && split1 < split2 && split2 < n_out)) return fail(C2KV_EINVAL, "need 0 < split1 < split2 < n_out");
  }
  if (!aligned16(x) || !aligned16(w)) return fail(C2KV_EINVAL, "x and w must be 16-byte aligned");
  const size_t need = c2kv_linear_workspace_size(tokens, n_out);
  if (workspace_bytes < need) return fail(C2KV_EINVAL, "workspace too small: need " + std::to_string(need) + " bytes");
  unsigned* err = nullptr;
  int sms = 0;
  c2kv_status s = device_state(&err, &sms);
  if (s != C2KV_OK) return s;
  const int n_pad = (tokens + 15) / 16 * 16;
  LinearParams p;
  std::memset(&p, 0, sizeof(p));
  s = encode_map(&p.tm_w, w, 2, (uint64_t)k_in, (uint64_t)n_out, 0, 0, 128);
  if (s != C2KV_OK) return s;
  s = encode_map(&p.tm_x, x, 2, (uint64_t)k_in, (uint64_t)tokens, 0, 0, (uint32_t)n_pad);
  if (s != C2KV_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.residual = static_cast<const __nv_bfloat16*>(residual);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.y2 = static_cast<__nv_bfloat16*>(y2);
  p.y3 = static_cast<__nv_bfloat16*>(y3);
  p.counters = reinterpret_cast<int32_t*>(ws);
  p.part = reinterpret_cast<float*>(ws + kLinearCountersBytes);
  p.err = err;
  p.tokens = tokens;
  p.n_pad = n_pad;
  p.k_in = k_in;
  p.n_out = n_out;
  p.split1 = split1;
  p.split2 = split2;
  p.stages = linear_stages(n_pad);
  p.epi = epilogue;
  p.cs = linear_plan_cs(n_out, k_in, n_pad, linear_ctas(sms));
  const int ctas = p.cs > 0 ? (n_out / 128) * p.cs : linear_ctas(sms);
  C2KV_LAUNCH(launch_linear(p, ctas, (flags & C2KV_LINEAR_OVERLAP_PREVIOUS) != 0, static_cast<cudaStream_t>(stream)));
  return C2KV_OK;
}

c2kv_status c2kv_rmsnorm(const void* x, int32_t tokens, int32_t dim, const void* w, float eps, void* y,
                         uint32_t flags, void* stream) {
  if (flags & ~uint32_t(C2KV_LINEAR_OVERLAP_PREVIOUS)) return fail(C2KV_EINVAL, "unknown rmsnorm flags");
  if (tokens < 1 || dim < 8 || dim % 8 != 0) return fail(C2KV_EINVAL, "need tokens >= 1 and dim a multiple of 8");
  if (!(eps > 0.f)) return fail(C2KV_EINVAL, "eps must be > 0");
  if (!x || !w || !y) return fail(C2KV_EINVAL, "null pointer");
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return fail(C2KV_EINVAL, "pointers must be 16-byte aligned");
  c2kv_status s = device_state(nullptr, nullptr);
  if (s != C2KV_OK) return s;
  C2KV_LAUNCH(launch_rmsnorm(static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w),
                           static_cast<__nv_bfloat16*>(y), tokens, dim, eps, (flags & C2KV_LINEAR_OVERLAP_PREVIOUS) != 0,
                           static_cast<cudaStream_t>(stream)));
  return C2KV_OK;
}

c2kv_status c2kv_test_expire_next_waits(int32_t n_launches) {
  if (n_launches < 0) return fail(C2KV_EINVAL, "n_launches < 0");
  g_inject_timeouts.store(n_launches);
  return C2KV_OK;
}

c2kv_status c2kv_kernel_launches(uint64_t* count) {
  if (count == nullptr) return fail(C2KV_EINVAL, "count is null");
  *count = g_kernel_launches.load(std::memory_order_relaxed);
  return C2KV_OK;
}

c2kv_status c2kv_device_error(int32_t* code) {
  if (code == nullptr) return fail(C2KV_EINVAL, "code is null");
  unsigned w = 0;
  C2KV_CUDA(cudaDeviceSynchronize());
  C2KV_CUDA(cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w)));
  const unsigned zero = 0;
  C2KV_CUDA(cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)));
  *code = (w & kErrTimeout) ? C2KV_ETIMEOUT : (w & kErrLength) ? C2KV_EDEVICE : C2KV_OK;
  return C2KV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without caller-provided scratch.
//
// c2kv_attend_decode needs a device scratch buffer for its split-K partial
// results.  Some callers cannot hand one over: a plugin whose host framework
// passes it only a stream and the tensors it owns and forbids allocating
// while work is being enqueued, or a serving loop that fixes every device
// allocation at start-up and may not call cudaMalloc (or any allocator that
// might) once it is running.  For them this entry point keeps the scratch in
// one fixed-size array in the library's own device memory.
// ---------------------------------------------------------------------------
namespace {

// 4 MiB per device, held from the moment the library's device code is loaded
// on a GPU until the process exits.
constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

uint8_t* g_noalloc_ptr[kMaxDevices] = {};   // device address of the array, per device
std::mutex g_noalloc_mu;

// Looks up the array's device address once per device (with that device
// current).  In host code the array's name is only a stand-in for the symbol,
// never an address a kernel may be given.
c2kv_status noalloc_scratch(uint8_t** out) {
  int dev = 0;
  C2KV_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(C2KV_EINVAL, "device index out of range");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    C2KV_CUDA(cudaGetSymbolAddress(&ptr, g_noalloc_scratch));
    if (ptr == nullptr) return fail(C2KV_ECUDA, "cudaGetSymbolAddress returned no address for the fixed scratch");
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return C2KV_OK;
}

}  // namespace

extern "C" c2kv_status c2kv_attend_decode_noalloc(const c2kv_geometry* geom, int32_t layer, int32_t batch,
                                                  void* const* k_caches, void* const* v_caches,
                                                  const void* const* rope_tables, int32_t cap,
                                                  const int32_t* n_cached_dev, int32_t max_keys, const void* q,
                                                  const void* k_new, const void* v_new, void* out, void* stream) {
  // The same argument checks as c2kv_attend_decode, done before anything is
  // enqueued (the counter clear below included).
  c2kv_status s = check_geom(geom);
  if (s != C2KV_OK) return s;
  if (layer < 0 || layer >= geom->n_layers) return fail(C2KV_EINVAL, "layer out of range");
  s = check_caches(batch, k_caches, v_caches, cap);
  if (s != C2KV_OK) return s;
  if (!n_cached_dev || !rope_tables) return fail(C2KV_EINVAL, "n_cached_dev / rope_tables is null");
  if (max_keys < 1 || max_keys > cap) return fail(C2KV_EINVAL, "max_keys must be in [1, cap]");
  if (!q || !k_new || !v_new || !out) return fail(C2KV_EINVAL, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new))
    return fail(C2KV_EINVAL, "q / k_new / v_new must be 16-byte aligned");
  for (int b = 0; b < batch; ++b)
    if (rope_tables[b] == nullptr || !aligned16(rope_tables[b])) return fail(C2KV_EINVAL, "bad rope table pointer");
  int sms = 0;
  s = device_state(nullptr, &sms);
  if (s != C2KV_OK) return s;
  const AttnWs w = attn_workspace(geom, batch, 1, max_keys, sms);
  if (w.total > kNoallocScratchBytes)
    return fail(C2KV_EINVAL, "this decode needs " + std::to_string(w.total) +
                                 " bytes of scratch, more than the fixed " +
                                 std::to_string(kNoallocScratchBytes) +
                                 " bytes of c2kv_attend_decode_noalloc; use c2kv_attend_decode with a workspace");
  uint8_t* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != C2KV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left in it; the arrival
  // counters must start at zero, the partial results need no clearing.
  if (w.tc || w.num_splits > 1) C2KV_CUDA(cudaMemsetAsync(scratch + w.counters_off, 0, w.counters_bytes, st));
  return c2kv_attend_decode(geom, layer, batch, k_caches, v_caches, rope_tables, cap, n_cached_dev, max_keys, q,
                            k_new, v_new, out, scratch, kNoallocScratchBytes, 0, stream);
}
