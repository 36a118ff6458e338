/*
 * b2pa.h -- C ABI of a batched paged-KV context (prefill) attention library
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one the FlashInfer API reference describes for
 * flashinfer.prefill.trtllm_batch_context_with_kv_cache (parameter list:
 * query, kv_cache, block_tables, seq_lens, max_q_len, max_kv_len,
 * bmm1_scale, bmm2_scale, cum_seq_lens_q, cum_seq_lens_kv, window_left,
 * kv_layout, sinks, out).  For every request b with q_len = cum_q[b+1] -
 * cum_q[b] query tokens and kv_len = seq_lens[b] keys, query i (0 <= i <
 * q_len) sits at position pos = kv_len - q_len + i (the queries are the
 * last q_len tokens of the sequence, as the TokenSpeed trtllm backend's
 * _init_extend_metadata builds them) and sees keys j with lo <= j <= pos,
 * lo = 0 if window_left < 0 else max(0, pos - window_left).  Query head h
 * reads kv head h / (H / Hkv).  With s_j = bmm1_scale * <q, K_j> and
 * m = max_j s_j:
 *
 *   out = bmm2_scale * sum_j e^{s_j - m} V_j / (sum_j e^{s_j - m} + [sinks] e^{sinks[h] - m})
 *
 * Key j of request b is slot j % page_size of page block_tables[b][j /
 * page_size] (TensorRT-LLM teardown (6), "Attention Backend 的 prepare()
 * 内部", section "句柄到偏移的物理含义": the table holds page ids and the
 * kernel adds id x page stride to the pool base).
 *
 * The library also does the step that precedes the attention in a serving
 * engine: writing the new tokens' K and V into the pools (b2pa_append_kv,
 * quantising to e4m3 for an FP8 cache).
 *
 * Conventions for every entry point:
 *  - All tensors are described by b2pa_tensor: a pointer, a dtype, a rank,
 *    and shape/stride arrays in ELEMENTS.  Tensors are owned by the caller;
 *    the library never frees or keeps them past the call.
 *  - Device tensors live on the current CUDA device; all work is enqueued on
 *    `stream` in stream order.  Entry points that return results to the host
 *    (b2pa_debug_worklist, b2pa_get_device_status) synchronise that stream.
 *  - Return value: B2PA_OK (0) or a negative b2pa_status.  Argument errors
 *    are detected on the host before anything is enqueued.  Problems that
 *    only the device can see (a malformed request, a page id outside the
 *    pool, a wait that timed out) never trap: the kernels skip the affected
 *    work and OR a bit into a device error word, which
 *    b2pa_get_device_status reads and clears.
 *  - Thread safety: calls on different streams use separate workspaces and
 *    may run concurrently; calls on one stream are ordered by the stream.
 */
#ifndef B2PA_H
#define B2PA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define B2PA_API __attribute__((visibility("default")))
#else
#define B2PA_API
#endif

/* cudaStream_t without pulling in the CUDA headers */
typedef struct CUstream_st* b2pa_stream_t;

enum b2pa_dtype {
    B2PA_BF16 = 1,      /* bfloat16 */
    B2PA_FP8_E4M3 = 2,  /* OCP FP8 E4M3 (float8_e4m3fn) */
    B2PA_FP32 = 3,
    B2PA_INT32 = 4
};

/* Which dims of a 4-D pool are page_size and num_kv_heads
 * (FlashInfer API reference, parameter kv_layout). */
enum b2pa_layout {
    B2PA_HND = 0, /* [num_pages, num_kv_heads, page_size, head_dim] */
    B2PA_NHD = 1  /* [num_pages, page_size, num_kv_heads, head_dim] */
};

enum b2pa_status {
    B2PA_OK = 0,
    B2PA_ERR_INVALID_ARG = -1, /* null pointer, bad rank/shape/dtype/stride, H % Hkv != 0, ... */
    B2PA_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. a forced kernel path that cannot run the shape) */
    B2PA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed; see b2pa_last_error_message */
    B2PA_ERR_DEVICE = -4       /* b2pa_get_device_status: the device error word was non-zero */
};

/* Bits of the device error word (b2pa_get_device_status). */
enum b2pa_device_error {
    B2PA_DEV_BAD_REQUEST = 1,   /* q_len < 0, q_len > kv_len, q_len > max_q_len, kv_len > max_kv_len,
                                   ceil(kv_len / page_size) > max_pages, or cum_q outside [0, num_tokens];
                                   that request's rows are not written */
    B2PA_DEV_BAD_PAGE = 2,      /* a page id a request reads is outside [0, num_pages); those keys read as 0 */
    B2PA_DEV_TIMEOUT = 4,       /* a pipeline wait in a kernel gave up; the call's output is undefined */
    B2PA_DEV_BAD_CUM_KV = 8,    /* cum_kv[b+1] - cum_kv[b] != seq_lens[b] (checked only where cum_kv is read) */
    B2PA_DEV_OVERFLOW = 16,     /* more work items than the workspace holds (cannot happen for valid bounds) */
    B2PA_DEV_BAD_SLOT = 32,     /* b2pa_append_kv: a cache_loc entry outside [0, num_pages * page_size);
                                   that token is not written */
    B2PA_DEV_BAD_SCALE = 64     /* b2pa_context_attention_tensor_scales: the device bmm1_scale is not
                                   finite and > 0, or bmm2_scale is not finite; nothing is written */
};

/* Kernel paths (b2pa_set_kernel_path). */
enum b2pa_path {
    B2PA_PATH_AUTO = 0,    /* tensor-core path when the shape allows it, else the generic path */
    B2PA_PATH_TCGEN05 = 1, /* TMA + tcgen05 tensor-core path only; B2PA_ERR_UNSUPPORTED if the shape does not fit */
    B2PA_PATH_GENERIC = 2  /* CUDA-core path for any shape */
};

typedef struct {
    void* data;         /* device pointer (host pointer where an entry point says so) */
    int32_t dtype;      /* enum b2pa_dtype */
    int32_t ndim;       /* 1..5 */
    int64_t shape[5];   /* extents, outermost first */
    int64_t stride[5];  /* strides in elements, outermost first */
} b2pa_tensor;

/*
 * b2pa_context_attention -- batched context attention over a paged KV cache.
 *
 * Arguments (all device tensors):
 *  q             [T, H, D] bf16; the ragged query tokens of all requests, request b
 *                owning rows cum_q[b] .. cum_q[b+1]-1.  stride[2] must be 1.
 *  k_pool,v_pool 4-D pools, same shape and dtype (bf16 or fp8 e4m3): [N, Hkv, P, D]
 *                (B2PA_HND) or [N, P, Hkv, D] (B2PA_NHD); any strides with stride[3] == 1.
 *                A single [N, 2, ...] cache is passed as its two strided views.
 *  block_tables  [B, max_pages] int32, stride[1] == 1.  Entries past
 *                ceil(seq_lens[b] / P) are never read.
 *  seq_lens      [B] int32, kv length per request (cached prefix + new tokens).
 *  cum_q         [B+1] int32, exclusive prefix sum of the query lengths.
 *  cum_kv        [B+1] int32, exclusive prefix sum of seq_lens.  Not needed for
 *                paged addressing; may be NULL.
 *  max_q_len     upper bound on every q_len (sizes the work list).
 *  max_kv_len    upper bound on every kv_len.
 *  bmm1_scale    factor on Q K^T (e.g. k_scale / sqrt(D)); finite and > 0.
 *  bmm2_scale    factor on the normalised P V (e.g. v_scale); finite.
 *  window_left   -1 for full causal attention, else W >= 0: keys pos-W .. pos.
 *  sinks         NULL, or [H] fp32: per query head, a logit (same units as
 *                bmm1_scale * q.k) whose exponential joins the denominator.
 *  layout        B2PA_HND or B2PA_NHD.
 *  out           [T, H, D] bf16, caller allocated, stride[2] == 1.  Only rows of
 *                valid requests are written.
 *  stream        CUDA stream (NULL = legacy default stream).
 *
 * No host synchronisation.  Allocates (cudaMalloc) only when this stream's
 * workspace must grow; once grown, the call can be captured in a CUDA graph.
 * On the tensor-core path the call is one kernel launch: every CTA sorts the
 * work items itself at its start, and the first CTA to claim the job writes
 * the list that the CTAs share after their first item (the stream's
 * workspace holds it, with four counter words that each launch leaves at
 * zero).  Calls on one stream must not overlap on the GPU, which stream order
 * guarantees.
 */
B2PA_API int b2pa_context_attention(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                           const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens,
                           const b2pa_tensor* cum_q, const b2pa_tensor* cum_kv, int32_t max_q_len,
                           int32_t max_kv_len, float bmm1_scale, float bmm2_scale, int32_t window_left,
                           const b2pa_tensor* sinks, int32_t layout, b2pa_tensor* out,
                           b2pa_stream_t stream);

/*
 * b2pa_context_attention_ragged -- b2pa_context_attention with the ragged
 * page table instead of a [B, max_pages] block table: FlashInfer's
 * paged_kv_indices / paged_kv_indptr / paged_kv_last_page_len (TensorRT-LLM
 * teardown (6), "Attention Backend 的 prepare() 内部", section "三条路径之二:
 * FlashInferAttentionMetadata——page table 三件套").  The page ids of all
 * requests are concatenated into one flat array, so a batch of short and long
 * requests carries no padding columns.
 *
 *  paged_kv_indices        int32 [nnz], contiguous: the page ids of request b
 *                          are paged_kv_indices[indptr[b] .. indptr[b+1]), in
 *                          logical order (key j on page j / P, slot j % P).
 *  paged_kv_indptr         int32 [B + 1], contiguous, non-decreasing from
 *                          indptr[0] (normally 0); B = its length - 1.
 *  paged_kv_last_page_len  int32 [B], contiguous: valid tokens of request b's
 *                          last page, in [1, P] when it has pages.
 * Request b's kv length is (indptr[b+1] - indptr[b] - 1) * P +
 * last_page_len[b] (0 without pages); it replaces seq_lens, and cum_kv is not
 * taken.  A request with a decreasing indptr or a last_page_len outside
 * [1, P] sets B2PA_DEV_BAD_REQUEST and its rows are not written.  The kv
 * lengths are derived on the device into the stream's workspace (B int32).
 * Every other argument, the layout rules and the errors are those of
 * b2pa_context_attention.
 */
B2PA_API int b2pa_context_attention_ragged(const b2pa_tensor* q, const b2pa_tensor* k_pool,
                           const b2pa_tensor* v_pool, const b2pa_tensor* paged_kv_indices,
                           const b2pa_tensor* paged_kv_indptr, const b2pa_tensor* paged_kv_last_page_len,
                           const b2pa_tensor* cum_q, int32_t max_q_len, int32_t max_kv_len, float bmm1_scale,
                           float bmm2_scale, int32_t window_left, const b2pa_tensor* sinks, int32_t layout,
                           b2pa_tensor* out, b2pa_stream_t stream);

/*
 * b2pa_batch_decode -- attention for a decode batch: every request has the
 * same number of query tokens, q_len_per_req, the last ones of its sequence.
 * This is the sibling call flashinfer.decode.trtllm_batch_decode_with_kv_cache
 * that the TokenSpeed trtllm backend makes in forward_decode (query,
 * kv_cache, block_tables, seq_lens, max_seq_len, bmm1_scale, bmm2_scale,
 * window_left, sinks, q_len_per_req; q_len_per_req > 1 for speculative
 * verification).  Query row i (0 <= i < q_len_per_req) of request b sits at
 * position seq_lens[b] - q_len_per_req + i and sees keys as in
 * b2pa_context_attention; the formula is the same.
 *
 * Arguments (device tensors) as for b2pa_context_attention, except:
 *  q, out         [B * q_len_per_req, H, D] bf16: request b owns rows
 *                 b * q_len_per_req .. (b + 1) * q_len_per_req - 1 (there is no
 *                 cum_q and no cum_kv).
 *  q_len_per_req  >= 1.
 *  max_seq_len    upper bound on every seq_lens[b] (sizes the split below).
 * A request with seq_lens[b] < q_len_per_req would have query rows with no
 * visible key (the TokenSpeed backend clamps its seq_lens to avoid that,
 * _clamped_spec_seqlens): it sets B2PA_DEV_BAD_REQUEST and its rows are not
 * written.
 *
 * Few query rows per request cannot fill the GPU with one work item per
 * request and kv head, so on the tensor-core path each request's kv range is
 * cut into chunks (about two work items per SM over the batch's longest
 * possible rows); the chunks' partial outputs go to the stream's workspace and
 * a second kernel merges them.  Allocation, capture and error behaviour are
 * those of b2pa_context_attention (the workspace also holds the partial rows:
 * B * q_len_per_req * H * chunks * (D + 2) fp32).
 */
B2PA_API int b2pa_batch_decode(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                           const b2pa_tensor* block_tables, const b2pa_tensor* seq_lens, int32_t q_len_per_req,
                           int32_t max_seq_len, float bmm1_scale, float bmm2_scale, int32_t window_left,
                           const b2pa_tensor* sinks, int32_t layout, b2pa_tensor* out, b2pa_stream_t stream);

/*
 * b2pa_context_attention_tensor_scales -- b2pa_context_attention with
 * bmm1_scale and bmm2_scale given as device tensors instead of host floats.
 * The FlashInfer API reference types both as "float | Tensor": a serving
 * engine that computes its FP8 scales on the GPU (k_scale, v_scale folded in,
 * as the TokenSpeed backend's _compute_scales does) passes them without a
 * device-to-host copy and without synchronising.
 *
 *  bmm1_scale, bmm2_scale   fp32 device tensors of one element (ndim 0 or 1),
 *                           4-byte aligned, read by the kernels in stream
 *                           order.  bmm1_scale * log2(e) is formed in double
 *                           and rounded once, exactly as the host-float entry
 *                           point does, so both give identical outputs for
 *                           identical scale values.
 * Every other argument, the layout rules and the errors are those of
 * b2pa_context_attention.  A device bmm1_scale that is not finite and > 0, or
 * a bmm2_scale that is not finite, cannot be seen on the host: the kernels
 * then write nothing and set B2PA_DEV_BAD_SCALE in the stream's device error
 * word.
 */
B2PA_API int b2pa_context_attention_tensor_scales(const b2pa_tensor* q, const b2pa_tensor* k_pool,
                           const b2pa_tensor* v_pool, const b2pa_tensor* block_tables,
                           const b2pa_tensor* seq_lens, const b2pa_tensor* cum_q, const b2pa_tensor* cum_kv,
                           int32_t max_q_len, int32_t max_kv_len, const b2pa_tensor* bmm1_scale,
                           const b2pa_tensor* bmm2_scale, int32_t window_left, const b2pa_tensor* sinks,
                           int32_t layout, b2pa_tensor* out, b2pa_stream_t stream);

/*
 * b2pa_context_attention_noalloc -- the same attention, for callers that must
 * not have the library allocate GPU memory.  The pages describe no such entry
 * point; it is an addition of this library.
 *
 * Who needs it: a serving engine that reserves nearly all of HBM for its KV
 * pool at start-up, and a framework whose own allocator accounts for every
 * byte, cannot let a library call cudaMalloc behind its back: the call could
 * fail once memory is taken, or break the caller's budget.
 * b2pa_context_attention grows a per-stream workspace with cudaMalloc on
 * first use; this entry point calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Its scratch (error word, work-distribution words and the work list) is a
 * fixed array inside the library: 256 B + 65536 work items x 16 B = 1 MiB +
 * 256 B, held on every GPU that loads the library until the process exits.
 * A call whose bounds need more than 65536 work items (batch x kv heads x
 * ceil(max_q_len / (2 * 128 / (H / Hkv)))) is rejected with
 * B2PA_ERR_INVALID_ARG and a message saying so; use b2pa_context_attention
 * for those.
 *
 * Arguments and results are those of b2pa_context_attention, plus:
 *  dev_status    NULL, or a caller-owned device uint32 that receives this
 *                call's device error word (b2pa_device_error bits) in stream
 *                order.  b2pa_get_device_status does not see this entry
 *                point's errors.
 * Only the tensor-core path runs here: a shape it cannot take returns
 * B2PA_ERR_UNSUPPORTED (b2pa_query_path tells beforehand).  The timing events
 * of b2pa_set_timing_events are not recorded by this entry point.
 *
 * The first call on a device looks up the scratch's device address there
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Every call on a device shares the one scratch array, which keeps the last
 * call's contents; the call clears the error word itself.  Calls whose
 * kernels overlap on the GPU (on different streams, or from different host
 * threads) race on the scratch and give undefined results: serialise them.
 */
B2PA_API int b2pa_context_attention_noalloc(const b2pa_tensor* q, const b2pa_tensor* k_pool,
                           const b2pa_tensor* v_pool, const b2pa_tensor* block_tables,
                           const b2pa_tensor* seq_lens, const b2pa_tensor* cum_q, const b2pa_tensor* cum_kv,
                           int32_t max_q_len, int32_t max_kv_len, float bmm1_scale, float bmm2_scale,
                           int32_t window_left, const b2pa_tensor* sinks, int32_t layout, b2pa_tensor* out,
                           uint32_t* dev_status, b2pa_stream_t stream);

/*
 * b2pa_debug_worklist -- build the work list of the tensor-core path (with a
 * kernel that runs the same sort as the attention kernel's start) and copy it
 * to the host (synchronises `stream`).
 *
 * Items are 4 int32 each: request b, kv head, item index it, cost.  Item it
 * of request b covers query tokens [it * n_qtiles * rows_per_tile, ...) and
 * cost = (kv tiles its rows touch) * (non-empty query tiles), sorted by
 * min(cost, cost_cap) descending, ties in (b, it, kv head) order.
 * geometry_out (may be NULL) receives {rows_per_tile, n_qtiles, kv_tile,
 * cost_cap}.  host_items_out holds cap items; *n_out gets the count (which
 * may exceed cap: only the first cap are copied).  Arguments as for
 * b2pa_context_attention; k_pool supplies P, Hkv, D and dtype.
 */
B2PA_API int b2pa_debug_worklist(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* block_tables,
                        const b2pa_tensor* seq_lens, const b2pa_tensor* cum_q, int32_t max_q_len,
                        int32_t max_kv_len, int32_t window_left, int32_t layout, int32_t* host_items_out,
                        int32_t cap, int32_t* n_out, int32_t* geometry_out, b2pa_stream_t stream);

/*
 * b2pa_debug_gather -- copy the first seq_lens[b] logical K and V tokens of
 * every request into contiguous k_out / v_out [sum(seq_lens), Hkv, D]
 * (same dtype as the pools) at row offset cum_kv[b], through the same
 * tensor-map page loads the attention kernel uses (the TensorRT-LLM Vanilla
 * backend's _gather_paged_kv, TensorRT-LLM teardown (6), section
 * "三条路径之一：VanillaAttention").  Requires a shape the tensor-core path
 * supports (else B2PA_ERR_UNSUPPORTED).  cum_kv is required; k_out/v_out
 * must be contiguous device tensors.
 */
B2PA_API int b2pa_debug_gather(const b2pa_tensor* k_pool, const b2pa_tensor* v_pool, const b2pa_tensor* block_tables,
                      const b2pa_tensor* seq_lens, const b2pa_tensor* cum_kv, int32_t layout,
                      b2pa_tensor* k_out, b2pa_tensor* v_out, b2pa_stream_t stream);

/*
 * b2pa_debug_gather_ragged -- b2pa_debug_gather for the ragged page table
 * (see b2pa_context_attention_ragged): the first kv_len(b) tokens of every
 * request, their pages found through the same shared addressing as the
 * attention kernel's loads, to k_out / v_out at row offset cum_kv[b].
 */
B2PA_API int b2pa_debug_gather_ragged(const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                      const b2pa_tensor* paged_kv_indices, const b2pa_tensor* paged_kv_indptr,
                      const b2pa_tensor* paged_kv_last_page_len, const b2pa_tensor* cum_kv, int32_t layout,
                      b2pa_tensor* k_out, b2pa_tensor* v_out, b2pa_stream_t stream);

/*
 * b2pa_append_kv -- write new tokens' K and V into the paged pools: the step
 * before the attention (TokenSpeed trtllm backend, _save_kv_and_prepare_q,
 * which calls fused_fp8_set_kv_buffer(k, v, k_cache, v_cache, cache_loc,
 * k_scale, v_scale, page_size) for an e4m3 cache and set_kv_buffer otherwise).
 *
 *   k_new, v_new     bf16 [T, Hkv, D] device tensors: token n's K and V rows.
 *                    head_dim contiguous; token and head strides multiples of
 *                    8 elements; 16-byte aligned; equal shapes and strides.
 *   k_pool, v_pool   the pools and layout exactly as for b2pa_context_attention
 *                    (bf16 or e4m3; Hkv and D must match k_new); their page,
 *                    head and slot strides must be multiples of 8 elements and
 *                    their bases 16-byte aligned.  Written in place.
 *   cache_loc        int32 [T] device tensor: token n goes to page
 *                    cache_loc[n] / page_size, slot cache_loc[n] % page_size.
 *                    Slots should be distinct; where two tokens name one slot,
 *                    which of them lands is unspecified.  A slot outside
 *                    [0, num_pages * page_size) is skipped and sets
 *                    B2PA_DEV_BAD_SLOT in the stream's device error word.
 *   k_scale, v_scale used by an e4m3 pool only, which stores x / scale (one
 *                    binary32 division) rounded to the nearest e4m3 value, ties
 *                    to even, magnitudes above 448 saturating to 448; a bf16
 *                    pool stores the bf16 bits unchanged.  Finite and > 0.
 *   D must be a multiple of 8.  T = 0 is a no-op.
 *
 * Asynchronous on `stream`; the caller owns every buffer.  The pages print
 * this call's interface, not its kernel; the rounding and saturation above
 * are this library's reading.
 */
B2PA_API int b2pa_append_kv(const b2pa_tensor* k_new, const b2pa_tensor* v_new, const b2pa_tensor* k_pool,
                            const b2pa_tensor* v_pool, const b2pa_tensor* cache_loc, float k_scale, float v_scale,
                            int32_t layout, b2pa_stream_t stream);

/*
 * b2pa_get_device_status -- synchronise `stream`, read and clear the device
 * error word of that stream's workspace.  Returns B2PA_OK if it was zero,
 * else B2PA_ERR_DEVICE with the bits (enum b2pa_device_error) in *bits_out
 * (may be NULL).
 */
B2PA_API int b2pa_get_device_status(b2pa_stream_t stream, uint32_t* bits_out);

/* Choose the kernel path for later calls in this process (enum b2pa_path). */
B2PA_API int b2pa_set_kernel_path(int32_t path);

/* Which path b2pa_context_attention would take for these shapes (enum b2pa_path), or a negative status. */
B2PA_API int b2pa_query_path(const b2pa_tensor* q, const b2pa_tensor* k_pool, const b2pa_tensor* v_pool,
                    const b2pa_tensor* out, int32_t layout);

/* Failure detection (no counterpart on the pages): the longest a pipeline wait
 * inside the tensor-core attention kernel may take, in ns of the GPU's global
 * timer, for later calls in this process; 0 restores the default, 2 s.  A wait
 * that runs out raises B2PA_DEV_TIMEOUT in the device error word: the CTA
 * stops, lets its in-flight copies and MMAs finish (those drains keep the 2 s
 * limit), frees its tensor memory and exits, so the context stays usable and
 * the call's output is undefined.  Serving code leaves the default. */
B2PA_API int b2pa_set_wait_limit_ns(uint64_t limit_ns);

/* Failure-detection tests (no counterpart on the pages): with on != 0, the
 * attention kernels of later calls in this process make one pipeline wait on a
 * barrier that nothing ever arrives on, so the wait limit runs out and every
 * CTA takes the abort path described at b2pa_set_wait_limit_ns; 0 turns it
 * off.  Nothing faults, traps or hangs: the call returns, the stream's device
 * error word holds B2PA_DEV_TIMEOUT and the context stays usable. */
B2PA_API int b2pa_debug_inject_stall(int32_t on);

/* Turn on (1) / off (0) the extra device-side input checks: page ids against the pool and
 * cum_kv against seq_lens.  Off by default. */
B2PA_API int b2pa_set_debug_checks(int32_t on);

/* Instrumentation (no counterpart on the pages): when both are non-NULL, later
 * b2pa_context_attention calls (that entry point only) on the tensor-core path record start_event just
 * before and stop_event just after launching the attention kernel, on the call's
 * stream, so a caller can time that kernel alone.  The arguments are cudaEvent_t
 * handles owned by the caller; NULL, NULL turns recording off. */
B2PA_API int b2pa_set_timing_events(void* start_event, void* stop_event);

/* Human-readable name of a b2pa_status. */
B2PA_API const char* b2pa_status_string(int32_t status);

/* Text of the last host-side error in this thread (empty if none). */
B2PA_API const char* b2pa_last_error_message(void);

/* Free every workspace this library allocated (all devices, all streams).  Must not be called while
 * work that uses them is in flight. */
B2PA_API void b2pa_release(void);

#ifdef __cplusplus
}
#endif

#endif /* B2PA_H */
