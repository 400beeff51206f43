/*
 * paged_mla.h -- C ABI of the GB300 (sm_103a) paged latent-MLA decode library.
 *
 * The operation is absorbed (latent) multi-head latent attention decode over a paged
 * FP8 KV cache with page size 1, as captured in "[Kimi-K3 MLA TP8] MLA performance"
 * (ROCm/aiter issue 4541), or with pages of 2^k tokens (k <= 10), the block-granular
 * addressing that issue's §5.2 proposes (page_size 128, the allocator's block):
 *   §2 "K3 MLA geometry": every cached token is one 576-wide latent entry (512 latent +
 *      64 rope) shared by all query heads; sm_scale = 1/sqrt(192).
 *   §3 "Entry point": the argument list of the decode call this ABI mirrors, with
 *      page_size = 1 and a single latent KV head.
 *   §4.1 / §4.2 argument tables: q and kv_buffer are float8_e4m3fn, q_scale and kv_scale
 *      are float32 scalars on the device, o is bfloat16 (tokens, heads, 512).
 *   §5.2: with page_size 1, kv_indptr holds per-request token counts (CSR), kv_indices
 *      one cache row id per token, kv_last_page_lens is all ones.  With page_size PS > 1
 *      (the paged-attention reading of the same arguments): kv_indptr counts pages,
 *      kv_indices holds one page id per page, kv_last_page_lens[b] in [1, PS] is the
 *      number of valid tokens in request b's last page.
 * and the partial-result merge of "Scaling Kimi K3 on AMD Instinct MI355X" §1 "Cache"
 * (decode context parallelism: partial answers carry normalisation information so that
 * a softmax-weighted merge is exact) and §4 "MLA" (history split into partitions).
 *
 * For request b, query token t < T_b = qo_indptr[b+1]-qo_indptr[b], head h:
 *   n_b   = kv_indptr[b+1] - kv_indptr[b]           (pages)
 *   L_b   = (n_b - 1) * PS + kv_last_page_lens[b]   (n_b > 0; 0 when n_b = 0;
 *                                                    = n_b when PS = 1)
 *   row_j = kv_buffer[kv_indices[kv_indptr[b] + j / PS]][j % PS]   (j < L_b)
 *   J     = { j : 0 <= j <= L_b - T_b + t }      (causal within the draft tokens;
 *                                                  every position when T_b = 1)
 *   s_j   = sm_scale * q_scale * kv_scale * sum_{d<576} q[r,h,d] * row_j[d]
 *   lse   = ln sum_{j in J} exp(s_j)
 *   o[c]  = kv_scale * sum_{j in J} exp(s_j - lse) * kv[row_j, c],   c < 512
 * with r = qo_indptr[b] + t.  An empty J gives o = 0 and lse = -inf.
 *
 * Conventions for every entry point
 *  - Ownership: the caller owns every buffer.  All tensor pointers are DEVICE pointers
 *    on the current CUDA device.  The library never allocates device memory; scratch
 *    comes from the caller's workspace (mla_decode_noalloc: from a fixed array inside the
 *    library).  It keeps only per-device caches of device attributes, kernel attributes
 *    and that array's address.
 *  - Asynchrony: work is enqueued on `stream` (NULL = legacy default stream) and the
 *    call returns without waiting, except mla_validate and mla_check_error, which
 *    synchronise `stream`.
 *  - Errors: every function returns an mla_status.  Argument errors are detected on the
 *    host before anything is enqueued.  Errors only visible on the device (an index
 *    outside the cache, an output row outside `o`, a pipeline wait that timed out) never
 *    fault or trap the GPU: the offending access is skipped and a bit is set in the
 *    workspace error word, read by mla_check_error.
 *  - Strides are in elements.
 */
#ifndef PAGED_MLA_H_
#define PAGED_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA runtime headers. */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
    MLA_DTYPE_FP8_E4M3FN = 1, /* 1-byte float8 e4m3fn codes */
    MLA_DTYPE_BF16 = 2,
    MLA_DTYPE_FP32 = 3,
    MLA_DTYPE_INT32 = 4
} mla_dtype_t;

/* A strided view of device memory.  shape/stride entries past ndim are ignored. */
typedef struct {
    void* ptr;
    int32_t ndim;      /* 0..4 (0 = scalar) */
    int32_t dtype;     /* mla_dtype_t */
    int64_t shape[4];
    int64_t stride[4]; /* in elements */
} mla_tensor_t;

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,         /* null pointer, wrong dtype/shape/stride, bad size */
    MLA_ERR_UNSUPPORTED = 2,         /* valid request outside what the kernels implement */
    MLA_ERR_WORKSPACE_TOO_SMALL = 3,
    MLA_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed */
    MLA_ERR_BAD_INDEX = 5,           /* device-side: index or indptr outside its buffer */
    MLA_ERR_TIMEOUT = 6,             /* device-side: a pipeline wait gave up (no fault) */
    MLA_ERR_BAD_INPUT = 7            /* mla_validate: indptr not monotone, kv_len < q_len,
                                        or kv_last_page_lens outside [1, page_size]
                                        (!= 1 for one-token pages) */
} mla_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_status_string(int status);

/*
 * Bytes of workspace mla_decode needs for a call with these sizes.
 *   batch_size    B (requests)
 *   num_heads     H (query heads per call: 12, 16, 96 ...)
 *   max_seqlen_q  largest T_b in the call (1 for plain decode)
 *   num_kv_splits <= 0: automatic split-KV scheduling; k >= 1: every request is split
 *                 into exactly k contiguous pieces of its positions (1 = never split)
 *   num_sms       SM count to plan for; <= 0 queries the current device.
 * The result is an upper bound for any call with the same (B, H, max_seqlen_q,
 * num_kv_splits) on that device.  The first 256 bytes of the workspace hold the device
 * error words and must be zero before first use (mla_check_error clears them again).
 */
int mla_get_workspace_size(int32_t batch_size, int32_t num_heads, int32_t max_seqlen_q,
                           int32_t num_kv_splits, int32_t num_sms, size_t* bytes_out);

/*
 * Latent-MLA decode.  The first 13 arguments follow the captured decode call (issue §3,
 * §4.1); the last three are this library's.
 *   q                 (sum_T, H, 576) FP8_E4M3FN, contiguous; 16-byte aligned.
 *   kv_buffer         (N_rows, 576), or (N_pages, PS, 1, 576) FP8_E4M3FN with PS a power
 *                     of two <= 1024 (PS = 1: one token a page); last dim contiguous,
 *                     token (slot) stride and page stride multiples of 16 bytes, pages not
 *                     overlapping; 16-byte aligned; N_pages * PS < 2^31.
 *   o                 (sum_T, H, 512) BF16 or FP32, last dim contiguous (written).
 *   qo_indptr         (B+1,) INT32: query-token CSR; qo_indptr[B] = sum_T.
 *   kv_indptr         (B+1,) INT32: page CSR (tokens when PS = 1).
 *   kv_indices        (n,) INT32 with n >= kv_indptr[B]; only [kv_indptr[0], kv_indptr[B])
 *                     is read.  Entries (page ids) must lie in [0, N_pages).
 *   kv_last_page_lens (B,) INT32: valid tokens of each request's last page, in [1, PS].
 *                     Required when PS > 1 (MLA_ERR_INVALID_ARG if NULL).  With PS = 1 it
 *                     may be NULL and must be all 1; values outside [1, PS] are clamped by
 *                     the decode and flagged by mla_validate only.
 *   max_seqlen_q      >= every T_b, 1..64.
 *   sm_scale          softmax scale (1/sqrt(192) for the captured model).
 *   q_scale, kv_scale 0-dim (or 1-element) FP32 device tensors: per-tensor dequant scales.
 *   num_kv_splits     see mla_get_workspace_size.
 *   lse_out           (sum_T, H) FP32 contiguous, or NULL (not written).
 *   workspace         device scratch of at least mla_get_workspace_size(...) bytes,
 *                     256-byte aligned, first 256 bytes zero before first use.
 * Device-side errors are reported through mla_check_error on the same workspace.
 * Calls that share a workspace must not overlap on the GPU.
 */
int mla_decode(const mla_tensor_t* q, const mla_tensor_t* kv_buffer, const mla_tensor_t* o,
               const mla_tensor_t* qo_indptr, const mla_tensor_t* kv_indptr,
               const mla_tensor_t* kv_indices, const mla_tensor_t* kv_last_page_lens,
               int32_t max_seqlen_q, float sm_scale, const mla_tensor_t* q_scale,
               const mla_tensor_t* kv_scale, int32_t num_kv_splits, const mla_tensor_t* lse_out,
               void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * Workspace for mla_decode_shared_prefix with these sizes (automatic split-KV); >= the
 * plain decode's.  Arguments as for mla_get_workspace_size.
 */
int mla_get_shared_prefix_workspace_size(int32_t batch_size, int32_t num_heads,
                                         int32_t max_seqlen_q, int32_t num_sms,
                                         size_t* bytes_out);

/*
 * mla_decode for a batch whose requests share their first cache positions: the prefix-
 * cache pattern of the captured concurrency-16/24 decode steps ("[Kimi-K3 MLA TP8] MLA
 * performance" §1 "Environment", §5.4 "Possible cross-request KV reuse").  Same
 * arguments and results as mla_decode with num_kv_splits = 0, except:
 *   shared_prefix_len  P >= 0: for every request b, its first P positions are the same
 *                      cache rows (with PS > 1: its first floor(P / PS) pages are the same
 *                      page ids), and every query sees all P positions
 *                      (P <= kv_len_b - q_len_b + 1).  With PS > 1 the cascade shares the
 *                      floor(P / PS) whole pages and leaves the rest to each request.  The caller knows this from its
 *                      prefix cache; it is not searched for.  A request breaking the
 *                      second condition is flagged (MLA_ERR_BAD_INPUT through
 *                      mla_check_error); breaking the first gives wrong results.
 *   workspace          at least mla_get_shared_prefix_workspace_size(...) bytes for the
 *                      shared-prefix path; with less (but at least
 *                      mla_get_workspace_size(B, H, max_seqlen_q, 0, ...)) it runs the
 *                      plain decode.
 * The shared positions are attended in groups of requests (96 query rows per tile, i.e.
 * 8 requests at 12 heads and q_len 1; 48 rows for batches of 4..7 requests of at most 24
 * rows), so each shared row is read once per group instead of once per request; each
 * request's own positions run separately and the two halves are merged by their
 * log-sum-exp.  Batches with fewer requests than one group, more than 48 query rows per
 * request, or fewer than 1024 shared positions (whole pages) run the plain decode.
 */
int mla_decode_shared_prefix(const mla_tensor_t* q, const mla_tensor_t* kv_buffer,
                             const mla_tensor_t* o, const mla_tensor_t* qo_indptr,
                             const mla_tensor_t* kv_indptr, const mla_tensor_t* kv_indices,
                             const mla_tensor_t* kv_last_page_lens, int32_t max_seqlen_q,
                             float sm_scale, const mla_tensor_t* q_scale,
                             const mla_tensor_t* kv_scale, int32_t shared_prefix_len,
                             const mla_tensor_t* lse_out, void* workspace,
                             size_t workspace_bytes, mla_stream_t stream);

/*
 * The CSR page table (kv_indptr, kv_indices) of a batch whose requests share their first
 * pages, built on the device from the compact form a prefix cache keeps: the shared pages
 * once and each request's own pages ("[Kimi-K3 MLA TP8] MLA performance" §1 "Environment":
 * decode batches over a shared prefix; §4.1: the page table mla_decode reads; §5.4:
 * cross-request reuse).  A caller that uploads its page table every step moves the shared
 * ids over the host link once instead of once per request, then calls
 * mla_decode_shared_prefix (or mla_decode) on the result.  For request b < B:
 *   kv_indptr[b]   = b * S + (own_indptr[b] - own_indptr[0]),   kv_indptr[B] likewise
 *   kv_indices[kv_indptr[b] + j] = shared_indices[j]                          (j < S)
 *                                = own_indices[own_indptr[b] + j - S]          (j >= S)
 *   shared_indices (S,) INT32 page ids (S >= 0; with S = 0 a null pointer is allowed)
 *   own_indptr     (B+1,) INT32, non-decreasing offsets into own_indices, own_indptr[0] >= 0
 *   own_indices    (>= own_indptr[B],) INT32 (empty: a null pointer is allowed)
 *   kv_indptr      (B+1,) INT32 (written)
 *   kv_indices     INT32 (written), room for B * S + own_indptr[B] - own_indptr[0] entries
 * All on the device; nothing is read by the host.  A request whose own_indptr entries are
 * out of order or past own_indices is skipped (its kv_indptr entry is not written) and
 * flags bit 2 in `error_word` (an int on the device, may be NULL); entries past the end of
 * kv_indices are not written and flag bit 8.  B <= 65535.  Enqueued on `stream`.
 */
int mla_expand_shared_prefix_indices(const mla_tensor_t* shared_indices,
                                     const mla_tensor_t* own_indptr,
                                     const mla_tensor_t* own_indices,
                                     const mla_tensor_t* kv_indptr, const mla_tensor_t* kv_indices,
                                     int32_t* error_word, mla_stream_t stream);

/*
 * Softmax-weighted merge of partial results ("Scaling Kimi K3 on AMD Instinct MI355X",
 * §1: each partial answer carries its normalisation, so shards merge exactly):
 *   for output row r < n_out and head h, over the partial rows
 *   P_r = reduce_idx[reduce_indptr[r] .. reduce_indptr[r+1]):
 *     M = max lse_parts[i,h];  w_i = exp(lse_parts[i,h] - M)
 *     o[r,h,:]   = sum w_i o_parts[i,h,:] / sum w_i
 *     lse[r,h]   = M + ln sum w_i
 *   Partials with lse = -inf weigh 0; if every partial is -inf (or P_r is empty) the
 *   row gets o = 0 and lse = -inf.
 *   o_parts        (P, H, 512) FP32, last dim contiguous
 *   lse_parts      (P, H) FP32, contiguous
 *   reduce_indptr  (n_out+1,) INT32;  reduce_idx (m,) INT32 entries in [0, P)
 *   o              (n_out, H, 512) BF16 or FP32, last dim contiguous (written)
 *   lse_out        (n_out, H) FP32 contiguous, or NULL
 * The reduce map lives on the device and is not read by the host; an entry outside
 * [0, P) is skipped and flagged in `error_word` (an int on the device, may be NULL).
 */
int mla_merge_partials(const mla_tensor_t* o_parts, const mla_tensor_t* lse_parts,
                       const mla_tensor_t* reduce_indptr, const mla_tensor_t* reduce_idx,
                       const mla_tensor_t* o, const mla_tensor_t* lse_out, int32_t* error_word,
                       mla_stream_t stream);

/*
 * The step after the decode: each head's 512-wide latent output mapped to v_head_dim = 128
 * by that head's matrix ("[Kimi-K3 MLA TP8] MLA performance" §2 geometry: kv_lora_rank
 * 512, v_head_dim 128, 12 heads a GPU; §3: a separate batched matmul after the decode):
 *   v[t, h, n] = sum_{k<512} o[t, h, k] * w_uv[h, k, n]
 * in fp32, rounded to bf16 (nearest even).
 *   o     (n_tok, H, 512) BF16 (mla_decode's o), last dim contiguous, token and head
 *         strides non-negative multiples of 8 elements, 16-byte aligned.
 *   w_uv  (H, 512, 128) BF16, contiguous, 16-byte aligned.
 *   v     (n_tok, H, 128) BF16, last dim contiguous, non-negative strides (written).
 * n_tok = 0 does nothing.  Shapes, dtypes, strides or alignments outside these return
 * MLA_ERR_INVALID_ARG before anything is enqueued.  Asynchronous on `stream`.
 */
int mla_latent_to_v(const mla_tensor_t* o, const mla_tensor_t* w_uv, const mla_tensor_t* v,
                    mla_stream_t stream);

/*
 * The step that produces the decode's inputs ("[Kimi-K3 MLA TP8] MLA performance" §3
 * "Entry point": q comes out of a fused step that rotates q's rope part, places it after
 * the 512 latent columns and writes the step's new cache entry into the cache the decode
 * reads; §2: an entry is 512 latent + 64 rope columns; §4.1: fp8 e4m3fn q and cache with
 * float32 per-tensor scales).  For token t < T and head h < H, with p = positions[t] and
 * the table row cos_sin[p] = (cos th_0 .. cos th_31, sin th_0 .. sin th_31):
 *   rot(v)  rotates the pairs of the 64 rope values v by th_i: pair i is (v[2i], v[2i+1])
 *           (is_neox = 0) or (v[i], v[i+32]) (is_neox = 1), and (x, y) becomes
 *           (x cos th_i - y sin th_i, y cos th_i + x sin th_i), every product and sum
 *           rounded to fp32 (no fused multiply-add);
 *   e(v, s) the e4m3fn code nearest to fp32(v / s) (ties to even, saturating at +-448);
 *   q_out[t, h, 0:512]   = e(q_nope[t, h, :], q_scale)
 *   q_out[t, h, 512:576] = e(rot(q_pe[t, h, :]), q_scale)
 *   cache slot slot_mapping[t] (= page * PS + slot) = [e(kv_c[t], kv_scale),
 *                                                     e(rot(k_pe[t]), kv_scale)]
 * so that the decode's dequantisation (code * scale) returns the rotated values.
 *   q_nope        (T, H, 512) BF16: the latent part of q (already absorbed)
 *   q_pe          (T, H, 64)  BF16: the rope part of q, before rotation
 *   kv_c          (T, 512)    BF16: the step's new latent entries
 *   k_pe          (T, 64)     BF16: their rope keys, before rotation
 *                 (each: last dim contiguous, 16-byte aligned, other strides non-negative
 *                 multiples of 8 elements: views into wider projections are fine)
 *   positions     (T,) INT32: position of each token (its row of cos_sin)
 *   cos_sin       (max_pos, 64) FP32, last dim contiguous, row stride a multiple of 4
 *   is_neox       0 or 1 (pair convention above)
 *   slot_mapping  (T,) INT32: cache slot of token t's entry; < 0: no entry (padding)
 *   q_scale, kv_scale  0-dim (or 1-element) FP32 device tensors
 *   q_out         (T, H, 576) FP8_E4M3FN, contiguous, 16-byte aligned (written): the
 *                 decode's q
 *   kv_buffer     the decode's cache, (N, 576) or (N_pages, PS, 1, 576) FP8_E4M3FN as
 *                 mla_decode takes it (written at the mapped slots only)
 *   error_word    device int32 (required): a slot >= N_pages * PS is skipped and sets bit
 *                 64; a position outside [0, max_pos) sets bit 1 and leaves that token's
 *                 rope columns (of q_out and of its entry) unwritten
 * Two tokens mapped to one slot race (which entry lands is unspecified); the outputs may
 * not overlap the inputs.  Shapes, dtypes, strides or alignments outside these return
 * MLA_ERR_INVALID_ARG before anything is enqueued.  Asynchronous on `stream`.
 */
int mla_qk_rope_concat_and_cache(const mla_tensor_t* q_nope, const mla_tensor_t* q_pe,
                                 const mla_tensor_t* kv_c, const mla_tensor_t* k_pe,
                                 const mla_tensor_t* positions, const mla_tensor_t* cos_sin,
                                 int32_t is_neox, const mla_tensor_t* slot_mapping,
                                 const mla_tensor_t* q_scale, const mla_tensor_t* kv_scale,
                                 const mla_tensor_t* q_out, const mla_tensor_t* kv_buffer,
                                 int32_t* error_word, mla_stream_t stream);

/*
 * Debug check of a decode call's index inputs on the device, then a host status:
 * MLA_OK, MLA_ERR_BAD_INPUT (indptr not monotone or not starting at 0 for qo, kv_len <
 * q_len, kv_last_page_lens outside [1, PS] (!= 1 when PS = 1), qo_indptr[B] != sum_T) or
 * MLA_ERR_BAD_INDEX (kv_indptr[B] beyond kv_indices, or an attended page id outside
 * [0, N_pages)).  Same arguments as
 * mla_decode minus the arithmetic ones.  Synchronises `stream`.
 */
int mla_validate(const mla_tensor_t* q, const mla_tensor_t* kv_buffer,
                 const mla_tensor_t* qo_indptr, const mla_tensor_t* kv_indptr,
                 const mla_tensor_t* kv_indices, const mla_tensor_t* kv_last_page_lens,
                 void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * Synchronises `stream`, returns the device-side errors recorded in the workspace's error
 * words since the last check (MLA_OK if none) and clears them: MLA_ERR_TIMEOUT before
 * MLA_ERR_BAD_INDEX (an index or indptr out of range), MLA_ERR_UNSUPPORTED (shared memory
 * misaligned) and MLA_ERR_BAD_INPUT (a shared prefix longer than a request's queries see).
 */
int mla_check_error(void* workspace, size_t workspace_bytes, mla_stream_t stream);

/*
 * Self-test of the bounded wait every decode pipeline role uses (no counterpart on the
 * pages: it exists so that the failure path of a wait can be exercised on the GPU without
 * a fault or a hang).  One thread initialises an mbarrier in shared memory that nothing
 * ever arrives at and waits on it with the library's wait, limited to limit_ns
 * (1 us .. 100 ms; the decode's own waits use 2 s).  The wait gives up when the limit
 * passes: it ORs the timeout bit into *error_word (the bit mla_check_error reports as
 * MLA_ERR_TIMEOUT), and the kernel writes result[0] = 1 if the wait returned success
 * (never expected), result[1] = the abort flag the wait raised (1), result[2] = the
 * microseconds spent waiting.  error_word (1 int32) and result (3 int32) are device
 * pointers.  Asynchronous on `stream`.
 */
int mla_selftest_bounded_wait(int32_t* error_word, int32_t* result, int64_t limit_ns,
                              mla_stream_t stream);

/* Size of the fixed device scratch array behind mla_decode_noalloc (16 MiB). */
#define MLA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * mla_decode without a workspace, for callers that cannot allocate device memory: code
 * living inside a framework whose device memory is owned by that framework's own
 * allocator, or a hook that is handed only its input and output tensors and has no way to
 * obtain scratch space.  (The pages have no counterpart of this entry point; it is part of
 * this library's interface only.)
 *
 * Arguments are those of mla_decode, minus workspace / workspace_bytes, plus:
 *   error_out  NULL, or a device int32 that receives this call's raw device error bits
 *              (0 = none; any other value is an error mla_check_error would report).
 *
 * Scratch: the split-KV partials and error words live in one file-scope device array of
 * MLA_NOALLOC_SCRATCH_BYTES, held by every GPU that loads the library until the process
 * exits.  A call whose mla_get_workspace_size(...) exceeds that returns
 * MLA_ERR_WORKSPACE_TOO_SMALL without enqueuing anything (on a 152-SM GPU the automatic
 * split fits up to ~350 requests with 12-16 heads and q_len 1, and ~18 requests with 12
 * heads and q_len 4; num_kv_splits = 1 fits any batch).  Nothing is allocated: the first call on each device looks up the array's
 * device address (so make that first call before any stream capture), and every call
 * runs all of mla_decode's host-side argument checks (returning their status with nothing
 * enqueued), then clears the array's error words and runs the ordinary decode on
 * `stream`.  Because each call clears the error words, the bits of a call are only kept
 * through its error_out: pass error_out to learn of index errors or timeouts.
 * All calls on a device share the array and it keeps the last call's contents: calls
 * that may overlap on the GPU (different streams without ordering) race on it.
 */
int mla_decode_noalloc(const mla_tensor_t* q, const mla_tensor_t* kv_buffer,
                       const mla_tensor_t* o, const mla_tensor_t* qo_indptr,
                       const mla_tensor_t* kv_indptr, const mla_tensor_t* kv_indices,
                       const mla_tensor_t* kv_last_page_lens, int32_t max_seqlen_q,
                       float sm_scale, const mla_tensor_t* q_scale, const mla_tensor_t* kv_scale,
                       int32_t num_kv_splits, const mla_tensor_t* lse_out, int32_t* error_out,
                       mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_MLA_H_ */
