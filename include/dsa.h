/*
 * dsa.h - C ABI of the GB300 (sm_103a) DeepSeek-Sparse-Attention hot path.
 *
 * The operations follow the sglang-jax DSA pages:
 *   "ref.py" (jnp reference implementations): build_index_share_map,
 *       streamindex_topk_ref, streamindex_page_topk_ref, sparse_mla_ref;
 *   "sparse_mla_prefill_qblock.py" (blocked sparse-MLA prefill):
 *       build_block_unit_tables, _qblock_kernel, sparse_mla_attention_qblock;
 *   "dsa_sparse_backend.py" (DSA sparse attention backend): IndexShare and the
 *       page budgets.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every tensor pointer is a DEVICE pointer owned by the caller,
 *           except where an argument is marked "host". The library allocates
 *           no memory: scratch space is a caller-provided workspace whose size
 *           the matching *_workspace_size() call reports.
 * Streams.  Every device entry point only enqueues kernels on `stream` (a
 *           cudaStream_t; NULL is the legacy default stream) and never
 *           synchronises, so calls may be captured in a CUDA graph.
 * dtypes.   bf16 tensors are passed as uint16_t (the raw bit pattern);
 *           metadata is int32.
 * Ragged batch metadata (identical for all calls, "D4" of the pages):
 *   seq_lens     [S]    kv length of request s, INCLUDING its new tokens;
 *   cu_q_lens    [S+1]  query-token offsets (cu_q_lens[S] == T);
 *   cu_kv_lens   [S+1]  cumulative page-aligned kv lengths; request s owns the
 *                       packed page-table entries starting at cu_kv_lens[s]/ps;
 *   page_indices [PTW]  physical page of every packed page-table entry, < P.
 *   Query token t of request s sits at absolute position
 *   pos(t) = seq_lens[s] - q_len(s) + (t - cu_q_lens[s]); it sees the key
 *   positions j with j < seq_lens[s] and j <= pos(t) (causal + kv_len mask).
 * Padding.  Unused index slots are -1. Selected sets are written in
 *           ascending index order.
 * Status.   Host-detected errors return a negative DSA_ERR_* code and enqueue
 *           nothing. Conditions detected on the device are OR-ed into the
 *           optional `dev_status` word (device int32, may be NULL): the
 *           offending access is skipped, never trapped.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

typedef void* dsa_stream_t; /* a cudaStream_t */

enum dsa_error {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARGUMENT = -1, /* null pointer, negative size, T != ... */
  DSA_ERR_UNSUPPORTED = -2,      /* a shape this build does not implement */
  DSA_ERR_WORKSPACE = -3,        /* workspace missing or too small */
  DSA_ERR_CUDA = -4,             /* a CUDA call or kernel launch failed */
  DSA_ERR_SHARED_BEFORE_FULL = -5,
  DSA_ERR_BAD_INDEXER_TYPE = -6,
  DSA_ERR_ALIGNMENT = -7,    /* a pointer is not 16-byte aligned */
  DSA_ERR_SCRATCH_LIMIT = -8 /* needs more than the built-in scratch of
                                dsa_sparse_mla_decode_noalloc (24 MiB) */
};

/* Bits OR-ed into *dev_status by the kernels. */
#define DSA_STATUS_UNION_TRUNCATED 0x1 /* a block's union exceeded u_max */
#define DSA_STATUS_BAD_METADATA 0x2    /* ragged metadata out of range */
#define DSA_STATUS_BAD_INDEX 0x4       /* a selected unit or page id out of range */
#define DSA_STATUS_TIMEOUT 0x8         /* a pipeline wait gave up (about 2 s) */
#define DSA_STATUS_INTERNAL 0x10       /* a launch-time invariant failed on the device */

/* ------------------------------------------------------------------------
 * IndexShare layer -> slot map (host only).
 * ref.py, build_index_share_map: a full layer (type 0) opens a new indexer
 * slot; a shared layer (type 1) consumes the slot of the nearest preceding
 * full layer and runs no indexer. types == NULL means every layer is full.
 * skip_offset is accepted and ignored, as on the page.
 *   types      host int32 [num_layers] (0 = full, 1 = shared) or NULL
 *   full_slot  host int32 [num_layers] out: slot of a full layer, -1 otherwise
 *   src_slot   host int32 [num_layers] out: slot whose top-k the layer uses
 *   num_full   host int32 out: number of full layers (= indexer key caches)
 * Errors: DSA_ERR_SHARED_BEFORE_FULL, DSA_ERR_BAD_INDEXER_TYPE.
 * ------------------------------------------------------------------------ */
DSA_API int dsa_index_build_share_map(const int32_t* types, int num_layers, int skip_offset, int32_t* full_slot,
                              int32_t* src_slot, int32_t* num_full);

/* ------------------------------------------------------------------------
 * Lightning indexer + exact token top-k.
 * ref.py, streamindex_topk_ref: s[t,j] = sum_h relu(q[t,h,:] . k[j,:]) * w[t,h]
 * accumulated in fp32 over the visible prefix j < min(seq_lens[s], pos(t)+1);
 * then the k highest-scoring visible positions, ties to the lower index
 * (exact: the pages' approximate top-k is not used).
 *   q        bf16 [T, Hi, Di]       indexer queries
 *   w        fp32 [T, Hi]           head weights (any scale folded in)
 *   kcache   bf16 [P, ps, Di]       paged indexer keys
 *   max_kv   upper bound of seq_lens (sizes the score workspace); a larger
 *            seq_len is clamped and flagged DSA_STATUS_BAD_METADATA
 *   topk     int32 [T, k] out       ascending positions, -1 padded
 *   topk_scores fp32 [T, k] out or NULL: the scores of `topk` (-inf on pads)
 *   ws/ws_bytes  workspace of dsa_indexer_workspace_size(T, S, max_kv, ps) bytes
 * Supported: Hi == 32, Di == 128, ps in {32, 64, 128}, 1 <= k.
 * ------------------------------------------------------------------------ */
DSA_API size_t dsa_indexer_workspace_size(int T, int S, int max_kv, int ps);
DSA_API int dsa_indexer_topk(dsa_stream_t stream, const uint16_t* q, const float* w, const uint16_t* kcache,
                     const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                     const int32_t* page_indices, int T, int S, int P, int PTW, int ps, int Hi, int Di, int max_kv,
                     int k, int32_t* topk, float* topk_scores, void* ws, size_t ws_bytes, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Lightning indexer + page top-k (and, optionally, the token top-k from the
 * same score pass).
 * ref.py, streamindex_page_topk_ref: the token scores are max-pooled per page
 * of ps positions (masked positions excluded), then the k_pages best pages
 * are kept (ties to the lower page); pages with no visible position are never
 * selected. Page ids are sequence-local; unused slots are -1.
 * The prefill budget of dsa_sparse_backend.py is k_pages = ceil(k / ps); the
 * decode page budget is min(budget, pages_per_seq).
 *   topk_pages  int32 [T, k_pages] out
 *   k, topk, topk_scores  as dsa_indexer_topk; topk == NULL skips the token
 *               top-k (k is then ignored).
 * ------------------------------------------------------------------------ */
DSA_API int dsa_indexer_page_topk(dsa_stream_t stream, const uint16_t* q, const float* w, const uint16_t* kcache,
                          const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                          const int32_t* page_indices, int T, int S, int P, int PTW, int ps, int Hi, int Di,
                          int max_kv, int k_pages, int32_t* topk_pages, int k, int32_t* topk, float* topk_scores,
                          void* ws, size_t ws_bytes, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Per-query-block union of selected units and the membership bitmap.
 * sparse_mla_prefill_qblock.py, build_block_unit_tables (plus the lift of
 * sparse_mla_attention_qblock's ragged mode): token t's sequence-local page
 * ids p >= 0 become global page-table keys g = cu_kv_lens[seq(t)]/ps + p
 * (cu_q_lens == NULL: ids are already global). T is padded to a multiple of
 * QB with empty rows. For block b:
 *   units   int32 [nQB, u_max]        ascending unique ids, -1 padded; a union
 *                                      larger than u_max keeps its u_max
 *                                      smallest ids and sets
 *                                      DSA_STATUS_UNION_TRUNCATED
 *   member  uint32 [nQB, u_max, QB/32] bit (q % 32) of word q/32 of slot u is
 *                                      1 iff query q of the block selected
 *                                      units[b, u] (slot-major, bit-packed)
 *   counts  int32 [nQB]               true (uncapped) union size
 * with nQB = ceil(T / QB). u_max <= 0 selects the lossless bound
 * min(QB * K, PTW); the outputs must then be sized with that value.
 *   topk_units int32 [T, K]  selected units per query, -1 padded
 * Supported: QB % 32 == 0, QB <= 1024. Needs no workspace.
 * ------------------------------------------------------------------------ */
DSA_API int dsa_build_block_union(dsa_stream_t stream, const int32_t* topk_units, int T, int K, int QB, int u_max,
                          const int32_t* cu_q_lens, const int32_t* cu_kv_lens, int S, int ps, int PTW,
                          int32_t* units, uint32_t* member, int32_t* counts, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Sparse absorbed-MLA attention over per-query selections (decode form).
 * ref.py, sparse_mla_ref: for query t and head h,
 *   o[t,h,:] = sum_j softmax_j(sm_scale * q[t,h,:Dk] . kv[j,:Dk]) kv[j,:Dv]
 * over the selected positions j that are visible (j < seq_len, j <= pos(t));
 * the value is the first Dv columns of the same latent row. A query with no
 * visible selected key outputs 0 (lse = -inf). Logits and softmax in fp32,
 * output rounded to bf16.
 *   q      bf16 [T, H, Dk]               [q_nope | q_rope]
 *   kv     bf16 [P, ps, row_stride]      [c_kv(Dv) | k_rope | pad]
 *   sel    int32 [T, K]  unit == 1: token positions; unit == ps: sequence-
 *                        local page ids (each expands to ps positions);
 *                        -1 entries are ignored, order does not matter
 *   o      bf16 [T, H, Dv] out
 *   lse    fp32 [T, H] out or NULL: natural-log sum of exp of the logits
 *   ws     workspace of dsa_sparse_mla_decode_workspace_size(T, H, Dv) bytes
 *          (split-key partials; 0 bytes needed when T*H is large)
 * Supported: Dk == 576, Dv == 512, row_stride in {576, 640}, ps in
 * {32, 64, 128}, H >= 1 (heads are processed 128 at a time).
 * Cache contents: with page units (and in the query-block and dense forms)
 * whole runs of 32 rows of each selected page are read and the rows past
 * the visible length are masked with a probability of exactly 0, so those
 * rows (the unwritten tail of a request's last page) must hold finite values
 * (0 x NaN is NaN), as in the pages' kernels; token units read only the
 * selected rows.
 * Reproducibility: every output is the same on every run: when a row's
 * keys are split across CTAs (few queries, long selections) the merging CTA
 * adds the splits in a fixed order, whichever CTA of the row finishes last.
 * ------------------------------------------------------------------------ */
DSA_API size_t dsa_sparse_mla_decode_workspace_size(int T, int H, int Dv);
DSA_API int dsa_sparse_mla_decode(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                          const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                          const int32_t* page_indices, const int32_t* sel, int K, int unit, int T, int S, int P,
                          int PTW, int ps, int H, int Dk, int Dv, float sm_scale, uint16_t* o, float* lse,
                          void* ws, size_t ws_bytes, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Sparse MLA decode without any allocation or caller workspace.
 * The source pages have no counterpart of this entry point. It is for
 * callers that cannot allocate device memory on this path: for example a
 * plugin that an inference engine hands only its input and output buffers,
 * or code that must not allocate once it is running. It computes the same
 * result as dsa_sparse_mla_decode (same arguments minus the workspace);
 * when the key list is split across CTAs, the split partials live in a
 * 24 MiB device array built into the library instead of a workspace.
 *  - Memory: nothing is allocated. The array is part of the library image,
 *    so every GPU that loads the library holds it until the process exits.
 *  - Set-up: the first call on a device looks up the array's address on that
 *    device; make that first call before any stream capture.
 *  - Sharing: all calls use the same array and leave their last contents in
 *    it (the merge counters are cleared on every call). Calls that overlap on
 *    the GPU (other streams, other host threads) race on the array, so
 *    serialise them.
 *  - Limit: a problem whose split scratch would exceed 24 MiB returns
 *    DSA_ERR_SCRATCH_LIMIT and enqueues nothing; use dsa_sparse_mla_decode
 *    with a workspace for it. Only devices 0..63 are served: on a device
 *    with a higher ordinal a call that needs the array returns DSA_ERR_CUDA.
 * ------------------------------------------------------------------------ */
DSA_API int dsa_sparse_mla_decode_noalloc(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv,
                                          int row_stride, const int32_t* seq_lens, const int32_t* cu_q_lens,
                                          const int32_t* cu_kv_lens, const int32_t* page_indices, const int32_t* sel,
                                          int K, int unit, int T, int S, int P, int PTW, int ps, int H, int Dk, int Dv,
                                          float sm_scale, uint16_t* o, float* lse, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Query-block sparse-MLA prefill over the block unions.
 * sparse_mla_prefill_qblock.py, _qblock_kernel / sparse_mla_attention_qblock:
 * query t of block b = t / QB walks the slots u < min(counts[b], u_max) of its
 * block; unit g = units[b,u] is physical page page_indices[g] whose row r is
 * key position kp = g*ps + r - (cu_kv_lens[seq(t)]/ps)*ps, visible iff the
 * membership bit of (u, t % QB) is set and kp <= pos(t) and kp < seq_len.
 * Same masked-softmax math and output as dsa_sparse_mla_decode with page
 * units (the pages' parity claim between the blocked and per-query kernels).
 *   units/member/counts  as written by dsa_build_block_union (same QB, u_max)
 *   o      bf16 [T, H, Dv] out; lse fp32 [T, H] out or NULL
 * Supported: as dsa_sparse_mla_decode. Needs no workspace.
 * ------------------------------------------------------------------------ */
DSA_API int dsa_sparse_mla_prefill_qblock(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                                  const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                                  const int32_t* page_indices, const int32_t* units, const uint32_t* member,
                                  const int32_t* counts, int QB, int u_max, int T, int S, int P, int PTW, int ps,
                                  int H, int Dk, int Dv, float sm_scale, uint16_t* o, float* lse,
                                  int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Query-block sparse-MLA prefill for a contiguous range of query tokens.
 * The pages have no counterpart of this entry point: it computes the rows
 * t_begin <= t < t_end of dsa_sparse_mla_prefill_qblock's output, with the
 * same arithmetic (bit for bit), and writes no other row. A caller that runs
 * one layer's attention in a few token ranges can start copying the finished
 * rows off the GPU while the later ranges compute.
 *   t_begin, t_end  0 <= t_begin <= t_end <= T (t_begin == t_end: nothing)
 *   every other argument as dsa_sparse_mla_prefill_qblock (q, o and lse keep
 *   their full [T, ...] extent; token t stays row t)
 * Errors: as dsa_sparse_mla_prefill_qblock; DSA_ERR_INVALID_ARGUMENT for a
 * range outside [0, T].
 * ------------------------------------------------------------------------ */
DSA_API int dsa_sparse_mla_prefill_qblock_range(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv,
                                                int row_stride, const int32_t* seq_lens, const int32_t* cu_q_lens,
                                                const int32_t* cu_kv_lens, const int32_t* page_indices,
                                                const int32_t* units, const uint32_t* member, const int32_t* counts,
                                                int QB, int u_max, int T, int S, int P, int PTW, int ps, int H,
                                                int Dk, int Dv, float sm_scale, int t_begin, int t_end, uint16_t* o,
                                                float* lse, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Approximate token top-k (the trade the pages make with approx_max_k on
 * their fast path; ref.py, streamindex_topk_ref is the exact definition).
 * Scores as dsa_indexer_topk. A row of n visible scores is folded into
 * B = min(n, over*k) bins (bin b holds positions b, b+B, b+2B, ...); each
 * bin keeps its largest score (lowest position on ties); the selection is
 * the exact top-k of the B bin maxima (ties to the lower bin), written as
 * ascending positions, -1 padded. count = min(k, n); over*k >= n makes it
 * the exact top-k up to ties; a larger `over` raises the recall.
 *   ws  workspace of dsa_indexer_topk_approx_workspace_size(T, S, max_kv,
 *       ps, k, over) bytes
 * Supported: as dsa_indexer_topk, k <= 16384, over >= 1.
 * ------------------------------------------------------------------------ */
DSA_API size_t dsa_indexer_topk_approx_workspace_size(int T, int S, int max_kv, int ps, int k, int over);
DSA_API int dsa_indexer_topk_approx(dsa_stream_t stream, const uint16_t* q, const float* w, const uint16_t* kcache,
                                    const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                                    const int32_t* page_indices, int T, int S, int P, int PTW, int ps, int Hi,
                                    int Di, int max_kv, int k, int over, int32_t* topk, void* ws, size_t ws_bytes,
                                    int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Dense causal absorbed-MLA attention: the route the backend takes for
 * layers without an indexer (dsa_sparse_backend.py, _run_dense, which calls
 * the dense ragged paged MLA kernel with the layer's sliding window and
 * logit soft cap; that kernel's module is not shown on the pages). For query
 * t every position j with j < seq_len, j <= pos(t) and, when
 * sliding_window > 0, j > pos(t) - sliding_window; with soft_cap > 0 each
 * logit l = sm_scale * q.k becomes soft_cap * tanh(l / soft_cap) before the
 * softmax. Output and lse as dsa_sparse_mla_decode.
 *   max_kv  an upper bound on seq_lens (host-known), sizes the key splits
 *   ws      workspace of dsa_sparse_mla_decode_workspace_size(T, H, Dv) bytes
 * Supported: as dsa_sparse_mla_decode; sliding_window >= 0, soft_cap >= 0.
 * ------------------------------------------------------------------------ */
DSA_API int dsa_dense_mla(dsa_stream_t stream, const uint16_t* q, const uint16_t* kv, int row_stride,
                          const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                          const int32_t* page_indices, int max_kv, int T, int S, int P, int PTW, int ps, int H,
                          int Dk, int Dv, float sm_scale, int sliding_window, float soft_cap, uint16_t* o,
                          float* lse, void* ws, size_t ws_bytes, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Paged write-back of the new tokens' rows into a paged cache: the step
 * directly before the indexer and the attention, which read these rows.
 * dsa_sparse_backend.py, _scatter_paged (and the Pallas paged_write_back of
 * sparse_mla_prefill_qblock.py): query token t of request s sits at position
 * pos(t) = seq_lens[s] - q_len(s) + (t - cu_q_lens[s]) and its row is copied
 * to row pos(t) % ps of physical page page_indices[cu_kv_lens[s]/ps +
 * pos(t)/ps]. Every other cache row is left untouched.
 *   rows   bf16 [T, src_stride]  the first D columns of row t are written
 *   cache  bf16 [P, ps, cache_stride]  updated in place; the first D columns
 *          of the destination rows are overwritten
 * Use it once per cache: D = 576 for the latent [c_kv | k_rope] cache
 * (cache_stride 576 or 640), D = 128 for the indexer key cache.
 * There are no padding rows in this ABI (T == cu_q_lens[S]), so no row is
 * sent to a sentinel page: a token whose destination falls outside the page
 * table or the pool sets DSA_STATUS_BAD_METADATA and is skipped.
 * Supported: D, src_stride, cache_stride multiples of 8 (16-byte rows),
 * D <= src_stride, D <= cache_stride, rows and cache 16-byte aligned.
 * Needs no workspace. Tokens write distinct rows whenever the metadata is
 * valid (positions of one request are distinct, requests own disjoint
 * page-table entries that map to distinct pages).
 * ------------------------------------------------------------------------ */
DSA_API int dsa_paged_write_back(dsa_stream_t stream, const uint16_t* rows, int src_stride, int D, uint16_t* cache,
                                 int cache_stride, const int32_t* seq_lens, const int32_t* cu_q_lens,
                                 const int32_t* cu_kv_lens, const int32_t* page_indices, int T, int S, int P,
                                 int PTW, int ps, int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Paged write-back into two caches that share one page table, in one launch
 * (no counterpart on the pages, which write each cache separately): a
 * layer's latent rows and, on a full layer, its indexer keys. Each token's
 * slot is found once; (rows0, src_stride0, D0, cache0, cache_stride0) and
 * (rows1, ...) follow the rules of dsa_paged_write_back, and both caches
 * hold P pages of ps rows. rows1 == cache1 == NULL with D1 == 0 writes the
 * first cache alone (dsa_paged_write_back is that call). Errors as
 * dsa_paged_write_back, for either target.
 * ------------------------------------------------------------------------ */
DSA_API int dsa_paged_write_back_pair(dsa_stream_t stream, const uint16_t* rows0, int src_stride0, int D0,
                                      uint16_t* cache0, int cache_stride0, const uint16_t* rows1, int src_stride1,
                                      int D1, uint16_t* cache1, int cache_stride1, const int32_t* seq_lens,
                                      const int32_t* cu_q_lens, const int32_t* cu_kv_lens,
                                      const int32_t* page_indices, int T, int S, int P, int PTW, int ps,
                                      int32_t* dev_status);

/* ------------------------------------------------------------------------
 * Token top-k -> page list, for the page-level decode shape of the pages.
 * dsa_sparse_backend.py, compute_topk_pages (k_pages_max = 512 there): per
 * query row, the ascending unique pages (position / ps) of the selected
 * tokens; the first `cap` of them are written, the rest of the row is -1.
 *   topk   int32 [T, K]  token positions, any order, -1 entries ignored
 *   pages  int32 [T, cap] out
 *   counts int32 [T] out or NULL: number of unique pages (not capped), so
 *          counts[t] > cap means row t was truncated
 * A position at or beyond max_pages * ps sets DSA_STATUS_BAD_INDEX and is
 * ignored. Supported: 1 <= max_pages <= 2^20, cap >= 1. Needs no workspace.
 * ------------------------------------------------------------------------ */
DSA_API int dsa_topk_pages_from_tokens(dsa_stream_t stream, const int32_t* topk, int T, int K, int ps,
                                       int max_pages, int cap, int32_t* pages, int32_t* counts,
                                       int32_t* dev_status);

/* Self-test of failure detection; the source pages have no counterpart.
 * Every pipeline wait in these kernels is bounded: when it runs out, the CTA
 * sets DSA_STATUS_TIMEOUT in the status word, unwinds and returns instead of
 * hanging or trapping. This entry runs one such wait on a barrier that
 * nothing arrives on, bounded by limit_clocks SM clocks (1 .. 1e10), so a
 * test can check that the status is set and the context stays usable.
 *   dev_status  device int32, required */
DSA_API int dsa_selftest_wait_timeout(dsa_stream_t stream, long long limit_clocks, int32_t* dev_status);

/* Number of streaming multiprocessors the kernels size their grids for
 * (device of the current context); a query helper, no device work. */
DSA_API int dsa_device_sm_count(void);

/* Number of kernels this process has enqueued through the library so far
 * (a host-side counter; a diagnostic, no device work). */
DSA_API long long dsa_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */
