/*
 * c2kv.h -- C ABI of the GB300 (sm_103a) C2KV composed-cache hot path.
 *
 * C2KV (compressed, composable, non-prefix KV-cache reuse) stores one
 * compressed, pre-RoPE K/V slot per k document tokens, keeps the stores in
 * host memory, and at request time streams the selected documents to the
 * GPU, re-applies RoPE at their new positions, concatenates them into one
 * cache and then prefills the question and decodes the answer over it.
 *
 * Sources (cited by page title and section):
 *   [EXPL]  "C 2 KV: Compressed and Composable KV Cache Reuse for Efficient
 *           LLM Inference", paper-daily.com explainer.  Sections used:
 *           "the problem" (它到底在解决什么问题？), "pipeline: extract, store,
 *           concatenate" (整体流程：抽取、存储、拼接), "C2 tokens"
 *           (C2 token：用额外的“记忆槽”承载压缩信息), "structured information flow"
 *           (为什么需要“结构化信息流”？), "positions at concatenation"
 *           (拼接时位置怎么处理？), "results" (实验结果：真的又快又准吗？).
 *   [ABS]   arXiv 2607.17715 listing (arxivdaily.com), English abstract.
 *
 * Conventions for every entry point:
 *   - No exception crosses the ABI; each call returns a c2kv_status and, on
 *     failure, c2kv_last_error() (thread-local) describes it.  All argument
 *     checks run on the host before anything is enqueued: a call that fails
 *     validation enqueues nothing.
 *   - All K/V/q tensors are bf16 (raw 16-bit patterns).  Device buffers are
 *     owned by the caller; the library never frees them.  Host inputs are
 *     read during the call only (copied where they must outlive it).
 *   - Device work is enqueued on the caller's `stream` (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream) and is ordered after the
 *     work already on it; calls return after enqueueing.
 *   - Cache layout per sequence: k_cache and v_cache are each
 *     [n_layers][n_kv_heads][cap][head_dim] bf16 (one contiguous key run per
 *     layer and kv head).  q head h reads kv head h / (n_q_heads/n_kv_heads).
 *   - RoPE is the rotate-half form with inv_freq_i = rope_theta^(-2i/d);
 *     angles are formed and reduced in fp64 (once per cache row, into a RoPE
 *     table); stored keys are rotated in double-float arithmetic on the fp32
 *     pipe and rounded once to bf16 (nearest even).
 *   - A kernel that finds a device-side problem (a bounded wait that expired,
 *     a device length beyond the cache capacity) records it in a device error
 *     word and skips the affected output; c2kv_device_error() reads it.
 */
#ifndef C2KV_H_
#define C2KV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct c2kv_store_s* c2kv_store;

typedef struct {
  int32_t n_layers;
  int32_t n_q_heads;
  int32_t n_kv_heads;   /* must divide n_q_heads; group = n_q/n_kv in {1,2,4,5,8} */
  int32_t head_dim;     /* 64 or 128 */
  double rope_theta;
} c2kv_geometry;

typedef enum {
  C2KV_OK = 0,
  C2KV_EINVAL = 1,     /* bad argument (null pointer, bad size, k mismatch, bad order) */
  C2KV_ENOMEM = 2,     /* pinned pool exhausted or host allocation failed */
  C2KV_ENOTFOUND = 3,  /* unknown document id */
  C2KV_ECAPACITY = 4,  /* composed or appended rows exceed the cache capacity */
  C2KV_ECUDA = 5,      /* a CUDA runtime call failed (message in c2kv_last_error) */
  C2KV_ETIMEOUT = 6,   /* a kernel's bounded wait expired (from c2kv_device_error) */
  C2KV_EDEVICE = 7,    /* a kernel rejected a device-side value (from c2kv_device_error) */
  C2KV_EIO = 8         /* a store file could not be opened, read or written */
} c2kv_status;

typedef enum {
  C2KV_MASK_CAUSAL = 0,      /* plain causal mask over the whole sequence */
  C2KV_MASK_STRUCTURED = 1,  /* [EXPL] "structured information flow" rules */
  C2KV_MASK_ANCHOR = 2       /* [EXPL] "results": the anchor-token ablation */
} c2kv_mask;

/* Thread-local description of the last failure on this thread ("" if none). */
const char* c2kv_last_error(void);

/* Library version string. */
const char* c2kv_version(void);

/*
 * Segment store: pinned host memory holding compressed pre-RoPE segments.
 * [EXPL] "the problem": the caches live in host memory and are moved to the
 * GPU when used; [EXPL] "positions at concatenation": they are kept before
 * RoPE so they can be re-rotated wherever they are composed.
 *
 * Creates a store on the current CUDA device with a pinned pool of
 * pinned_bytes (cudaHostAlloc), a non-blocking copy stream and events.
 * Returns C2KV_EINVAL for a bad geometry, C2KV_ENOMEM if the pool cannot be
 * pinned.  *out receives the handle (owned by the caller; free with
 * c2kv_store_destroy).
 */
c2kv_status c2kv_store_create(const c2kv_geometry* geom, size_t pinned_bytes,
                              c2kv_store* out);

/* Waits for the store's copies in flight, then frees the pool and handles. */
void c2kv_store_destroy(c2kv_store store);

/*
 * Copies n_docs compressed segments into the pinned pool.
 * [EXPL] "C2 tokens": one slot per k document tokens, only the slots' K/V
 * are kept.  For document i: doc_ids[i] (unique, not yet stored),
 * n_tokens[i] >= 1 original tokens, 1 <= n_slots[i] <= n_tokens[i] slots
 * stored at compression ratio k >= 1, and host pointers k_pre[i], v[i] to
 * bf16 arrays [n_layers][n_kv_heads][n_slots[i]][head_dim] (K before RoPE).
 * The inputs are copied; the caller keeps ownership.
 * Errors: C2KV_EINVAL (bad sizes, null pointer, duplicate id),
 * C2KV_ENOMEM (pool full; nothing of this call is stored).
 */
c2kv_status c2kv_store_segments(c2kv_store store, int32_t n_docs,
                                const int32_t* doc_ids, const int32_t* n_tokens,
                                const int32_t* n_slots, int32_t k,
                                const void* const* k_pre, const void* const* v);

/*
 * Persists the store.  [EXPL] "pipeline: extract, store, concatenate": each
 * document's compressed cache is extracted once, stored, and reused by any
 * later request; these two calls keep the stored caches across processes.
 *
 * c2kv_store_save writes every stored document (ascending ids: id, original
 * length, slots, k, then its K and V rows [n_layers][n_kv_heads][slot][d]
 * bf16) after a header holding the geometry, in host byte order, to `path`
 * (created or truncated).  Errors: C2KV_EINVAL (null argument), C2KV_EIO.
 *
 * c2kv_store_load adds the documents of such a file to `store`, which must
 * have the geometry the file was saved with.  Documents read before an error
 * stay in the store.  Errors: C2KV_EIO (cannot open, truncated), C2KV_EINVAL
 * (not a store file, another geometry, a bad record, an id already stored),
 * C2KV_ENOMEM (pool full).
 */
c2kv_status c2kv_store_save(c2kv_store store, const char* path);
c2kv_status c2kv_store_load(c2kv_store store, const char* path);

/* Looks up one stored document: its original length, slot count and k. */
c2kv_status c2kv_store_lookup(c2kv_store store, int32_t doc_id,
                              int32_t* n_tokens, int32_t* n_slots, int32_t* k);

/*
 * Host-only composition planner (no device work; usable without a GPU).
 * [EXPL] "positions at concatenation": documents are taken in composed
 * order, composed doc c = input doc order[c] (order NULL = identity; order
 * must be a permutation of 0..n_docs-1).  Each document occupies its
 * original length of positions, so composed doc c starts at position
 * pos_offset[c] = sum of n_tokens of the composed docs before it, and its
 * slots start at row slot_start[c] = sum of their n_slots.  Outputs (host,
 * n_docs entries each, may be NULL): slot_start, pos_offset; totals
 * *total_slots = sum n_slots and *total_tokens = sum n_tokens (the position
 * of the first appended question token).  Slot j of composed doc c sits at
 * pos_offset[c] + min((j+1)k, n_tokens) - 1.
 * Errors: C2KV_EINVAL (bad order, sizes, int32 overflow).
 */
c2kv_status c2kv_plan(int32_t n_docs, const int32_t* n_tokens,
                      const int32_t* n_slots, const int32_t* order,
                      int32_t* slot_start, int32_t* pos_offset,
                      int32_t* total_slots, int32_t* total_tokens);

/*
 * Composes one request's cache.  [EXPL] "pipeline": fetch the documents'
 * compressed caches, re-apply position encoding at their new positions and
 * concatenate them, with no repair step; [EXPL] "positions at
 * concatenation": slot j of composed doc c is rotated at
 * pos_offset[c] + min((j+1)k, n_tokens_c) - 1.
 *
 * doc_ids[n_docs] (repeats allowed), order as in c2kv_plan, k must equal the
 * k every document was stored with.  k_cache/v_cache: caller-owned device
 * buffers [n_layers][n_kv_heads][cap][head_dim] bf16; rows [0, N) of every
 * layer and kv head are written (N = total slots), rows >= N are untouched.
 * rope_table_out (required): caller-owned device buffer of
 * c2kv_rope_table_bytes(geom, cap) bytes receiving, for every cache row r,
 * the cos/sin of its position for the head_dim/2 RoPE frequencies as fp32
 * (hi, lo) pairs, layout [cap][head_dim/2][cos_hi, cos_lo, sin_hi, sin_lo].
 * Row r < N holds slot r's position; row r >= N holds L_tot + (r - N), the
 * position of the (r-N)-th token appended after the documents (reading: the
 * question starts right after the documents' original length L_tot).
 * Prefill and decode rotate with this table.
 * pos_dev_out: optional device int32 [cap] receiving the position of every row.
 * Host outputs (optional): *n_slots_out = N, *next_pos_out = L_tot.
 * The segments are copied host->device on the store's copy stream in layer
 * groups; the table and the re-rotation of each group run on `stream` (the
 * latter once its copy has landed), and all of it is ordered before later
 * work on `stream`.  The store must not be destroyed before that work
 * completes.
 * Errors: C2KV_EINVAL, C2KV_ENOTFOUND, C2KV_ECAPACITY (N > cap), C2KV_ECUDA.
 */
c2kv_status c2kv_compose(c2kv_store store, int32_t n_docs, const int32_t* doc_ids,
                         const int32_t* order, int32_t k, void* k_cache,
                         void* v_cache, int32_t cap, void* rope_table_out,
                         int32_t* pos_dev_out, int32_t* n_slots_out,
                         int32_t* next_pos_out, void* stream);

/*
 * c2kv_compose over the layers [layer_begin, layer_end) only, with flags:
 *
 * C2KV_COMPOSE_NO_REALIGN — the ablation of [EXPL] "results" that drops the
 *   position re-alignment: every document keeps the positions it was
 *   extracted at (slot j at min((j+1)k, n_c) - 1, no offset off_c), so all
 *   documents start at position 0.  Appended tokens still start at L_tot,
 *   the summed original length (reading: the ablation changes the
 *   documents' positions only).  c2kv_plan's pos_offset does not apply.
 *
 * C2KV_COMPOSE_CONTINUE — continue the composition started by the last
 *   c2kv_compose / c2kv_compose_layers call on this store into the same
 *   RoPE table (same doc_ids, order, k, flags other than this one, caches
 *   and cap): the table and pos_dev_out are not rebuilt, and the
 *   copies of these layers are queued behind that call's copies on the
 *   store's copy stream instead of waiting for the caller's stream.  So a
 *   caller can compose layer group 0, enqueue work on those layers (the
 *   question prefill), then compose group 1, and the prefill overlaps the
 *   later groups' host->device copies ([EXPL] "the problem": loading the
 *   cache is the dominant TTFT cost).  The caller guarantees that nothing
 *   issued on `stream` since the first call reads or writes rows [0, N) of
 *   the continued layers.  The re-rotation of the layers is ordered on
 *   `stream` after their copies.
 *
 * 0 <= layer_begin < layer_end <= n_layers.  Other arguments, outputs and
 * errors as c2kv_compose; C2KV_EINVAL also for a CONTINUE that does not
 * follow a composition of the same request (documents, k, flags, caches,
 * cap, table) on this store.  The store remembers the compositions into the
 * 1024 tables most recently composed into; a CONTINUE into an older one is
 * refused the same way.
 */
#define C2KV_COMPOSE_NO_REALIGN 1u
#define C2KV_COMPOSE_CONTINUE 2u
c2kv_status c2kv_compose_layers(c2kv_store store, int32_t n_docs, const int32_t* doc_ids,
                                const int32_t* order, int32_t k, uint32_t flags,
                                int32_t layer_begin, int32_t layer_end, void* k_cache,
                                void* v_cache, int32_t cap, void* rope_table_out,
                                int32_t* pos_dev_out, int32_t* n_slots_out,
                                int32_t* next_pos_out, void* stream);

/* Bytes of a RoPE table of `rows` rows: rows * (head_dim/2) * 16. */
size_t c2kv_rope_table_bytes(const c2kv_geometry* geom, int32_t rows);

/*
 * Builds a RoPE table (layout as in c2kv_compose) for arbitrary positions:
 * row r gets the cos/sin of position pos_dev[r] (device int32 [rows]), for
 * caches filled by other means than c2kv_compose.  Angles pos * inv_freq are
 * formed in fp64 and reduced mod 2*pi before the fp64 sincos.
 */
c2kv_status c2kv_rope_table(const c2kv_geometry* geom, const int32_t* pos_dev,
                            int32_t rows, void* table_out, void* stream);

/*
 * Device scratch (bytes) that c2kv_attend_prefill / c2kv_attend_decode /
 * c2kv_attend_masked need for `batch` sequences of `t_len` new tokens each,
 * with at most `max_keys` keys per sequence (cached + new).  The scratch
 * holds split-K partial results and per-(sequence, head) arrival counters;
 * it must be zeroed once before first use (c2kv_workspace_init) and may then
 * be reused by calls that do not overlap on the GPU.  Returns 0 on bad input.
 */
size_t c2kv_attend_workspace_size(const c2kv_geometry* geom, int32_t batch,
                                  int32_t t_len, int32_t max_keys);

/* Zeroes a workspace on `stream` (cudaMemsetAsync). */
c2kv_status c2kv_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * Question prefill for one layer of `batch` requests.
 * [EXPL] "pipeline": after composition the question is appended and
 * generation starts.
 *
 * k_caches[b], v_caches[b]: host array of device pointers to request b's
 * cache base (layer 0, layout as above); `layer` selects the layer.
 * rope_tables[b]: host array of device pointers to request b's RoPE table
 * (from c2kv_compose).  n_cached[b] (host): rows already in the cache.
 * q: device [batch][q_len][n_q_heads][head_dim] (before RoPE);
 * k_new, v_new: device [batch][q_len][n_kv_heads][head_dim] (k before RoPE).
 * Question token i lands at row n_cached[b] + i and is rotated with that
 * row of the table (q and k alike); then out[b][i] = softmax(q_i K^T /
 * sqrt(d)) V over the n_cached[b] + i + 1 visible keys (all cached rows plus
 * question tokens 0..i), written to device out [batch][q_len][n_q_heads]
 * [head_dim] bf16.  q_len > 1 runs QK^T and PV on the tcgen05 tensor cores.
 * workspace: device scratch of c2kv_attend_workspace_size(geom, batch,
 * q_len, max_b(n_cached[b] + q_len)) bytes, zeroed once.
 * Errors: C2KV_EINVAL, C2KV_ECAPACITY (n_cached[b] + q_len > cap), C2KV_ECUDA.
 */
c2kv_status c2kv_attend_prefill(const c2kv_geometry* geom, int32_t layer,
                                int32_t batch, void* const* k_caches,
                                void* const* v_caches, const void* const* rope_tables,
                                int32_t cap, const int32_t* n_cached, int32_t q_len,
                                const void* q, const void* k_new, const void* v_new,
                                void* out, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * One decode step for one layer of `batch` sequences.  [EXPL] "results":
 * each generated token reads the whole composed cache, which C2KV shrinks.
 *
 * As prefill with one new token per sequence, except that the lengths live
 * on the device so a captured sequence of calls can be replayed:
 * n_cached_dev[b] (device int32) rows are cached; the new token's key is
 * rotated with table row n_cached_dev[b], stored with its value at that row,
 * and the token attends over n_cached_dev[b] + 1 keys -- all in one kernel
 * launch.  max_keys (host) bounds n_cached_dev[b] + 1 for every b and sizes
 * the grid; a device length over max_keys or cap is recorded in the device
 * error word and that sequence's output is skipped.
 * q: [batch][n_q_heads][head_dim]; k_new, v_new: [batch][n_kv_heads]
 * [head_dim]; out: [batch][n_q_heads][head_dim].  The lengths are not
 * advanced (see c2kv_seq_advance).
 * workspace: c2kv_attend_workspace_size(geom, batch, 1, max_keys) bytes.
 */
c2kv_status c2kv_attend_decode(const c2kv_geometry* geom, int32_t layer,
                               int32_t batch, void* const* k_caches,
                               void* const* v_caches, const void* const* rope_tables,
                               int32_t cap, const int32_t* n_cached_dev, int32_t max_keys,
                               const void* q, const void* k_new, const void* v_new,
                               void* out, void* workspace, size_t workspace_bytes,
                               uint32_t flags, void* stream);

/*
 * Decode flag: the launch may begin while the kernel enqueued just before it
 * on `stream` is still finishing (programmatic dependent launch).  Before it
 * waits for that kernel it reads only n_cached_dev, the RoPE table and the
 * cache rows below n_cached_dev[b] of this layer, so the caller promises that
 * the previous kernel writes none of these (e.g. it is the decode of another
 * layer, or the projection producing q/k_new/v_new -- but not
 * c2kv_seq_advance).  q, k_new, v_new, out and the workspace are touched only
 * after the previous kernel has completed.
 */
#define C2KV_DECODE_OVERLAP_PREVIOUS 1u

/*
 * c2kv_attend_decode without a workspace argument: the paper has no
 * counterpart; this is a convenience of the library.
 *
 * For callers that cannot allocate device memory where they decode -- a
 * plugin whose host framework hands it only a stream and tensors and forbids
 * allocation while enqueueing, or a serving loop that freezes all device
 * allocations at start-up.  The split-K scratch lives instead in one
 * fixed-size array (4 MiB) in the library's device memory; every GPU that
 * loads the library holds that array until the process exits.  This call
 * allocates nothing (no cudaMalloc/cudaFree, no allocating library routine).
 *
 * Arguments and results are those of c2kv_attend_decode (with flags 0).  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  The
 * array is shared by every call and keeps the previous call's contents: each
 * call clears its arrival counters on `stream` first, so two calls whose GPU
 * work can overlap (for example calls on different streams) race on the
 * array; issue such calls one after the other.  A decode whose scratch would
 * exceed the array is rejected with C2KV_EINVAL before anything is enqueued.
 */
c2kv_status c2kv_attend_decode_noalloc(const c2kv_geometry* geom, int32_t layer,
                                       int32_t batch, void* const* k_caches,
                                       void* const* v_caches, const void* const* rope_tables,
                                       int32_t cap, const int32_t* n_cached_dev,
                                       int32_t max_keys, const void* q, const void* k_new,
                                       const void* v_new, void* out, void* stream);

/* Adds `delta` to n_cached_dev[b] for b < batch (device kernel). */
c2kv_status c2kv_seq_advance(int32_t batch, int32_t* n_cached_dev, int32_t delta,
                             void* stream);

/*
 * Attention over one extraction sequence under a mask (the "mask mode").
 * [EXPL] "structured information flow": n_doc document tokens followed by
 * n_slot slot tokens.  C2KV_MASK_STRUCTURED: document tokens keep the
 * causal mask and see no slot; slot i sees the sink block B(0) (document
 * tokens [0, k)), its own block [i*k, min((i+1)k, n_doc)) and slots 0..i.
 * [EXPL] "positions at concatenation": documents sit at 0..n_doc-1 and slot
 * i at min((i+1)k, n_doc) - 1.  C2KV_MASK_ANCHOR: the anchor-token
 * ablation of [EXPL] "results", read as a change of mask only: the n_slot
 * extra tokens take the slots' positions; document token r sees document
 * tokens 0..r and every extra token; extra token i sees every document
 * token and extra tokens 0..i.  C2KV_MASK_CAUSAL: plain causal attention,
 * token t at position t (n_slot must be 0).
 * q: device [N][n_q_heads][head_dim], kk, v: device [N][n_kv_heads][head_dim]
 * with N = n_doc + n_slot, all before RoPE; out: device [N][n_q_heads][d].
 * workspace: c2kv_attend_workspace_size(geom, 1, N, N) + c2kv_masked_extra_bytes
 * (geom, N) bytes (the sequence's RoPE table and its rotated keys and values
 * are staged there), zeroed once.
 */
c2kv_status c2kv_attend_masked(const c2kv_geometry* geom, int32_t mask,
                               int32_t n_doc, int32_t n_slot, int32_t k,
                               const void* q, const void* kk, const void* v,
                               void* out, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Extra scratch bytes c2kv_attend_masked needs beyond the attention scratch. */
size_t c2kv_masked_extra_bytes(const c2kv_geometry* geom, int32_t n_tokens);

/*
 * The synthetic-weight decoder step around the attention calls: its linear
 * layers and RMSNorm.  [EXPL] "the problem" (Fig. 1): the time to first token
 * and the decode rate of the whole model are what the cache reuse buys, and
 * a decoder layer runs these projections and its MLP around the attention
 * over the composed cache.
 *
 * c2kv_linear: y[t][n] = sum_k x[t][k] * w[n][k] on the tensor cores (fp32
 * accumulation, bf16 result) for t < tokens, then an epilogue:
 *   C2KV_LINEAR_STORE   y [tokens][n_out] = the product;
 *   C2KV_LINEAR_ADD     y [tokens][n_out] = product + residual [tokens][n_out]
 *                       (residual may be y: an in-place residual update);
 *   C2KV_LINEAR_SPLIT3  output columns [0, split1) to y [tokens][split1],
 *                       [split1, split2) to y2, [split2, n_out) to y3 (the
 *                       q, k and v of a fused QKV projection);
 *   C2KV_LINEAR_SWIGLU  rows 128i .. 128i+63 of w are the gate rows of
 *                       features 64i .. 64i+63 and rows 128i+64 .. 128i+127
 *                       their up rows; y [tokens][n_out / 2] =
 *                       silu(gate) * up, silu(g) = g / (1 + e^-g).
 * x: device bf16 [tokens][k_in], w: device bf16 [n_out][k_in] (row-major,
 * as a linear layer's weight), both 16-byte aligned.  1 <= tokens <= 256,
 * k_in a positive multiple of 64, n_out a positive multiple of 128 up to
 * 1048576.  workspace: c2kv_linear_workspace_size(tokens, n_out) bytes of
 * device memory, zeroed once (c2kv_workspace_init); calls of any shapes that
 * fit it may share it as long as their GPU work does not overlap (a launch
 * with C2KV_LINEAR_OVERLAP_PREVIOUS touches it only after the kernel before
 * it has completed).  flags: C2KV_LINEAR_OVERLAP_PREVIOUS lets the launch
 * begin, and request its first weight tiles, while the kernel before it on
 * `stream` finishes (the caller promises that kernel does not write w); x,
 * the residual and the outputs are touched only after it completes.
 * Errors: C2KV_EINVAL, C2KV_ECUDA.
 *
 * c2kv_rmsnorm: y[t] = x[t] / sqrt(mean_i x[t][i]^2 + eps) * w for t < tokens,
 * x and y device bf16 [tokens][dim], w bf16 [dim] (dim a multiple of 8,
 * 16-byte aligned pointers), sums in fp32.  flags as c2kv_linear.
 */
#define C2KV_LINEAR_STORE 0
#define C2KV_LINEAR_ADD 1
#define C2KV_LINEAR_SPLIT3 2
#define C2KV_LINEAR_SWIGLU 3
#define C2KV_LINEAR_OVERLAP_PREVIOUS 1u
size_t c2kv_linear_workspace_size(int32_t tokens, int32_t n_out);
c2kv_status c2kv_linear(const void* x, int32_t tokens, int32_t k_in, const void* w, int32_t n_out,
                        int32_t epilogue, const void* residual, void* y, void* y2, void* y3,
                        int32_t split1, int32_t split2, void* workspace, size_t workspace_bytes,
                        uint32_t flags, void* stream);
c2kv_status c2kv_rmsnorm(const void* x, int32_t tokens, int32_t dim, const void* w, float eps, void* y,
                         uint32_t flags, void* stream);

/*
 * Reads and clears the device error word of the current device (waits for
 * the device).  *code receives C2KV_OK, C2KV_ETIMEOUT or C2KV_EDEVICE; the
 * return value is C2KV_ECUDA only if the read itself failed.
 */
c2kv_status c2kv_device_error(int32_t* code);

/*
 * Kernel launches this library has enqueued in the process so far, counted
 * once each when the launch call succeeds (a launch enqueued while a stream
 * is being captured into a CUDA graph counts once, at capture, and not at
 * each replay).  Host-only; never fails except for a null count (C2KV_EINVAL).
 */
c2kv_status c2kv_kernel_launches(uint64_t* count);

/*
 * Test hook for the failure path (the pages have no counterpart): the next
 * n_launches decode launches (c2kv_attend_decode, c2kv_attend_decode_noalloc,
 * c2kv_attend_prefill with q_len 1) each wait, at their first key tile, on a
 * barrier nothing arrives on, for ~0.5 ms of GPU clock.  The wait expires and
 * the kernel takes its timeout path: it records C2KV_ETIMEOUT in the device
 * error word, lets its copies in flight land and returns; that launch's
 * outputs are undefined, the cache rows it appends are written, and the
 * context stays usable.  0 disarms it.  Process-wide; C2KV_EINVAL for n < 0.
 */
c2kv_status c2kv_test_expire_next_waits(int32_t n_launches);

#ifdef __cplusplus
}
#endif

#endif /* C2KV_H_ */
