/*
 * fd_attention.h -- C ABI of the GB300 (sm_103a) flash-decoding library.
 *
 * One decode step of attention: every sequence b of a batch contributes one
 * query token per query head, which attends over that sequence's cached
 * keys and values.  The cache is token-major and either contiguous (a
 * sequence owns a run of rows starting at kv_start_idx[b]) or paged (a block
 * table maps the sequence's logical pages to physical pages of a pool).
 * K and V are fp16, bf16 or FP8-e4m3 with one fp32 scale per tensor.
 *
 * The computation is split-KV partial attention with an online softmax
 * (running max, running sum, rescaled accumulator) followed by a
 * log-sum-exp merge of the partial states, for MHA, GQA and MQA head layouts.
 *
 * Passages that define the operation:
 *  - "From SGLang kernel source to GPU trace: DeepSeek V4.1 Flash-Decode",
 *    section 3.1: the decode kernel's arguments (q, FP8 k_cache/v_cache,
 *    output, kv_start_idx and seq_len per sequence, head count, head
 *    dimension, softmax scale, batch); section 2.2: FP8 KV converted inside
 *    the load stage, not by a separate pass;
 *  - "SGLang Prefill optimisation: dissecting FlashAttention kernel
 *    bottlenecks with GPU Trace", section 2.2: the online softmax loop
 *    (scores = dot(q, k) * scale, running max, rescale factor
 *    exp(m_old - m_new), running sum, accumulator update);
 *  - "Learn CUDA from scratch, chapter 15: GPU profiling and LLM inference",
 *    section 15.26: paged addressing (physical page from the block table,
 *    row = page * page_size + offset in a [page, offset, head, dim] pool);
 *    section 15.12: one pass over a KV head serves its group of
 *    QH / KVH query heads; section 15.13: a ragged batch scans each
 *    sequence's real length only.
 *
 * Conventions (readings where the pages are silent):
 *  - q and out are dense [batch, num_q_heads, head_dim]; lse is dense fp32
 *    [batch, num_q_heads];
 *  - contiguous K/V: [kv_rows, num_kv_heads, head_dim], kv_start_idx in rows;
 *    paged K/V: [num_pages, page_size, num_kv_heads, head_dim],
 *    block_table row-major [batch, block_table_stride] of int32 page ids;
 *  - query head qh reads KV head qh / (num_q_heads / num_kv_heads);
 *  - k = k_scale * stored(k), v = v_scale * stored(v) (pass 1.0 for 16-bit
 *    caches); score = softmax_scale * dot(q, k);
 *  - lse = natural log of sum_t exp(score_t); a sequence with seq_len 0
 *    gets out = 0 and lse = -inf;
 *  - out is rounded once, to nearest even, into q's dtype.
 *
 * Ownership and synchronisation: every pointer argument is device memory
 * owned by the caller (except where a function says "host").  The library
 * allocates, frees and synchronises nothing inside fd_decode_attention; all
 * of its work is enqueued on `stream`.  The workspace is caller-owned scratch
 * memory of at least fd_workspace_bytes(...) bytes; it holds no state that
 * the caller must keep between calls except the sticky device-error word
 * read by fd_check_device_error.  Calls that share one workspace must be
 * ordered on one stream.
 *
 * Devices and host threads: calls run on the CUDA device current in the
 * calling thread, and several devices may be used from one process.  The
 * library keeps, per device, the SM count and whether each kernel's
 * shared-memory limit has been raised, and per process a small cache of TMA
 * descriptors keyed by cache pointer and shape; all of these are guarded for
 * concurrent calls from several host threads.  They are kept for the life of
 * the process: do not use the library on a device after cudaDeviceReset.
 */
#ifndef FD_ATTENTION_H_
#define FD_ATTENTION_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as a cudaStream_t / CUstream (NULL = the legacy default stream). */
typedef struct CUstream_st *fd_stream_t;
/* Same object as a cudaEvent_t / CUevent. */
typedef struct CUevent_st *fd_event_t;

typedef enum {
  FD_OK = 0,
  FD_ERR_INVALID_ARG = 1,          /* bad pointer, size or layout; nothing launched */
  FD_ERR_UNSUPPORTED = 2,          /* valid but not implemented (head_dim, dtype pair, ...) */
  FD_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < fd_workspace_bytes(...) */
  FD_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed */
  FD_ERR_DEVICE_BOUNDS = 5,        /* a kernel met a cache row / page id out of range */
  FD_ERR_DEVICE_TIMEOUT = 6        /* a kernel's bounded wait expired */
} fd_status;

/* Element formats.  FD_I8 is a symmetric signed 8-bit code: the element's
 * value is the two's-complement integer (-128 .. 127) times its scales, no
 * zero point ("Learn CUDA from scratch, chapter 15", section 15.11: INT8 K/V
 * payloads with fp32 scales). */
typedef enum { FD_F16 = 0, FD_BF16 = 1, FD_E4M3 = 2, FD_I8 = 3 } fd_dtype;

/* Kernel selection for the split (partial attention) phase. */
typedef enum {
  FD_KERNEL_AUTO = 0,  /* FD_KERNEL_TC for one KV head with at least 64 query rows (query
                          heads times q_len), else FD_KERNEL_MMA where supported, else the
                          CUDA-core kernel */
  FD_KERNEL_SIMT = 1,  /* CUDA-core FMA kernel (every supported shape) */
  FD_KERNEL_MMA = 2,   /* tensor-core kernel with warp-level mma.sync products, operands
                          widened in registers; FD_ERR_UNSUPPORTED where it does not apply */
  FD_KERNEL_TC = 3,    /* tensor-core kernel with tcgen05 products (accumulators in tensor
                          memory, FP8 widened once per tile into shared memory): e4m3
                          caches, fp16 queries, head_dim 128, 17..128 query rows per KV
                          head (query heads per KV head times q_len), no per-token scales,
                          page sizes 8..256; FD_ERR_UNSUPPORTED elsewhere */
  FD_KERNEL_FMA = 4    /* the mma.sync kernel's TMA pipeline, plan and shapes with CUDA-core
                          FMA arithmetic instead of tensor cores (the comparison arm): e4m3
                          caches, head_dim 128, at most 8 query rows per KV head, KV heads a
                          multiple of 8, no per-token scales, page sizes of at least 8;
                          FD_ERR_UNSUPPORTED elsewhere; never chosen by FD_KERNEL_AUTO */
} fd_kernel;

/*
 * Scratch bytes fd_decode_attention needs for these sizes on the current
 * device (host function, no device work).  Returns 0 for invalid sizes.
 * The figure covers the partial (m, l, acc) states of the split phase, the
 * per-stream tile prefix of the split plan and a 256-byte header; it grows
 * with the device's SM count, not with sequence lengths.  For
 * fd_decode_attention_multi pass num_q_heads * q_len as num_q_heads.
 */
size_t fd_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim);

/*
 * One decode step of attention (see the file comment for the definition).
 *
 * q            [batch, num_q_heads, head_dim] of q_dtype (FD_F16 or FD_BF16).
 * k_cache, v_cache
 *              contiguous: [kv_rows, num_kv_heads, head_dim] of kv_dtype;
 *              paged: [kv_rows / page_size, page_size, num_kv_heads, head_dim].
 *              Base addresses 16-byte aligned.
 * kv_start_idx int32 [batch] first row of each sequence (contiguous mode), or NULL.
 * block_table  int32 [batch, block_table_stride] page ids (paged mode), or NULL.
 *              Exactly one of kv_start_idx / block_table is non-NULL.  Entries
 *              past ceil(seq_len[b] / page_size) are never read.
 * seq_len      int32 [batch] tokens per sequence (0 allowed; negative = 0).
 * kv_rows      number of token rows K and V hold (paged: pages * page_size).
 *              Rows outside [0, kv_rows) are never read: the kernel records
 *              FD_ERR_DEVICE_BOUNDS in the workspace and treats the token as
 *              absent.
 * num_q_heads, num_kv_heads
 *              num_q_heads % num_kv_heads == 0; group = num_q_heads / num_kv_heads <= 128.
 * head_dim     64 or 128.
 * page_size    paged mode: power of two in [1, 256]; contiguous mode: ignored.
 * softmax_scale, k_scale, v_scale
 *              finite fp32 factors (scores use softmax_scale * k_scale).
 * kv_dtype     FD_F16 (with q FD_F16), FD_BF16 (with q FD_BF16), FD_E4M3
 *              (OCP e4m3fn, with either q dtype) or FD_I8 (signed 8-bit
 *              codes, with either q dtype).
 * out          [batch, num_q_heads, head_dim] of q_dtype.
 * lse          fp32 [batch, num_q_heads], or NULL if not wanted.
 * workspace    device scratch of workspace_bytes >= fd_workspace_bytes(...),
 *              256-byte aligned.
 *
 * Returns FD_OK once the work is enqueued; argument errors return before any
 * launch.  Device-side index errors surface through fd_check_device_error.
 */
fd_status fd_decode_attention(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *kv_start_idx, const int32_t *block_table,
                              int block_table_stride, const int32_t *seq_len, int64_t kv_rows,
                              int batch, int num_q_heads, int num_kv_heads, int head_dim,
                              int page_size, float softmax_scale, float k_scale, float v_scale,
                              fd_dtype q_dtype, fd_dtype kv_dtype, void *out, float *lse,
                              void *workspace, size_t workspace_bytes, fd_stream_t stream);

/* Granularity of the finer K/V scales of fd_decode_attention_scaled. */
typedef enum {
  FD_SCALE_TENSOR = 0, /* none: k_scale / v_scale only                           */
  FD_SCALE_HEAD = 1,   /* one fp32 per KV head: k_scales[kvh]                     */
  FD_SCALE_TOKEN = 2   /* one fp32 per cache row and KV head: k_scales[row * KVH + kvh] */
} fd_scale_kind;

/*
 * fd_decode_attention with finer FP8 / INT8 scales ("Learn CUDA from scratch,
 * chapter 15", section 15.11: KV quantisation with a scale per tensor, per
 * head or per token).  The K and V elements of cache row `row` and KV head
 * `kvh` are decoded as
 *     k = k_scale * ks * dec(code),   v = v_scale * vs * dec(code),
 * with ks = k_scales[kvh], vs = v_scales[kvh] (FD_SCALE_HEAD) or
 * ks = k_scales[row * num_kv_heads + kvh], vs likewise (FD_SCALE_TOKEN; `row`
 * is the cache row of the token, contiguous or paged, the same index the
 * caches use).  FD_SCALE_TENSOR ignores both arrays and equals
 * fd_decode_attention.
 *
 * k_scales, v_scales  device fp32 arrays, 4-byte aligned: [num_kv_heads]
 *                     (FD_SCALE_HEAD) or [kv_rows * num_kv_heads]
 *                     (FD_SCALE_TOKEN); NULL only with FD_SCALE_TENSOR.
 * Finer scales need kv_dtype FD_E4M3 or FD_I8 (else FD_ERR_UNSUPPORTED).  Every other
 * argument, the workspace contract and the errors are those of
 * fd_decode_attention.
 */
fd_status fd_decode_attention_scaled(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *kv_start_idx, const int32_t *block_table,
                                     int block_table_stride, const int32_t *seq_len,
                                     int64_t kv_rows, int batch, int num_q_heads,
                                     int num_kv_heads, int head_dim, int page_size,
                                     float softmax_scale, float k_scale, float v_scale,
                                     fd_scale_kind scale_kind, const float *k_scales,
                                     const float *v_scales, fd_dtype q_dtype, fd_dtype kv_dtype,
                                     void *out, float *lse, void *workspace,
                                     size_t workspace_bytes, fd_stream_t stream);

/*
 * Decode attention for q_len query tokens per sequence (a speculative-decoding
 * verify batch, "Learn CUDA from scratch, chapter 15", section 15.21: the
 * target model checks q_len drafted tokens in one pass).  The last q_len
 * tokens of each sequence are the new ones and are already in the cache
 * (seq_len counts them): query token j (0 <= j < q_len) sits at position
 * seq_len[b] - q_len + j and attends to keys 0 .. seq_len[b] - q_len + j, its
 * own and every earlier one (causal among the new tokens), with the
 * definition of fd_decode_attention.  A query with no key (seq_len[b] <
 * q_len - j) gets out = 0 and lse = -inf.
 *
 * q, out  [batch, num_q_heads, q_len, head_dim] of q_dtype (head-major: the
 *         q_len tokens of one head are adjacent rows).
 * lse     fp32 [batch, num_q_heads, q_len], or NULL.
 * q_len   1 .. 16, with (num_q_heads / num_kv_heads) * q_len <= 128 (else
 *         FD_ERR_UNSUPPORTED); q_len = 1 equals fd_decode_attention_scaled.
 * workspace_bytes >= fd_workspace_bytes(batch, num_q_heads * q_len, ...).
 * Every other argument as for fd_decode_attention_scaled.
 */
fd_status fd_decode_attention_multi(const void *q, const void *k_cache, const void *v_cache,
                                    const int32_t *kv_start_idx, const int32_t *block_table,
                                    int block_table_stride, const int32_t *seq_len,
                                    int64_t kv_rows, int batch, int q_len, int num_q_heads,
                                    int num_kv_heads, int head_dim, int page_size,
                                    float softmax_scale, float k_scale, float v_scale,
                                    fd_scale_kind scale_kind, const float *k_scales,
                                    const float *v_scales, fd_dtype q_dtype, fd_dtype kv_dtype,
                                    void *out, float *lse, void *workspace,
                                    size_t workspace_bytes, fd_stream_t stream);

/*
 * KV-cache append of one new token per sequence ("Learn CUDA from scratch,
 * chapter 15", section 15.9: cache write layouts, contiguous and paged, and
 * the single-token decode append; quantisation with the scales of section
 * 15.11; n_new > 1: the drafted tokens of a speculative verify step,
 * section 15.21).  For every sequence b with positions[b] >= 0, every new
 * token i < n_new and every KV head h, with t = positions[b] + i, the row
 * r = kv_start_idx[b] + t (contiguous) or
 * block_table[b][t / page_size] * page_size + t % page_size (paged) of K
 * receives k_new[b][i][h][0 .. head_dim), and V likewise:
 *   16-bit cache (kv_dtype == new_dtype): the elements as they are;
 *   8-bit cache (FD_E4M3 or FD_I8), QMAX = 448 or 127, s the element's scale:
 *     s = k_scale                                  FD_SCALE_TENSOR
 *       = k_scale * k_scales[h]                    FD_SCALE_HEAD
 *       = k_scale * ks,  ks = amax / (QMAX * k_scale), stored to
 *         k_scales[r * num_kv_heads + h], amax = max_d |k_new[b][i][h][d]|
 *         (ks = 1 when amax = 0)                   FD_SCALE_TOKEN
 *     code = e4m3: nearest to x / s, ties to even, |x / s| > 448 -> 448;
 *            int8: nearest integer to x / s, ties to even, clamped to +-127.
 *   Each product and quotient above is one IEEE fp32 operation.
 *
 * k_new, v_new  [batch, n_new, num_kv_heads, head_dim] of new_dtype (FD_F16
 *               or FD_BF16), 16-byte aligned, device.
 * n_new         new tokens per sequence, 1 .. 16.
 * k_cache, v_cache, kv_start_idx, block_table, block_table_stride, kv_rows,
 * page_size     as for fd_decode_attention; the caches are written.
 * positions     int32 [batch] device: the first new token's index in its
 *               sequence; < 0 leaves the sequence alone.  The block table
 *               must cover positions[b] + n_new - 1.  Rows outside [0, kv_rows) or
 *               negative page ids are not written and are recorded as
 *               FD_ERR_DEVICE_BOUNDS (fd_check_device_error).
 * k_scale, v_scale  finite; > 0 for 8-bit caches.
 * scale_kind, k_scales, v_scales  as for fd_decode_attention_scaled; with
 *               FD_SCALE_TOKEN the arrays are written at the appended rows.
 * workspace     >= 256 bytes, 256-byte aligned (the device error word); the
 *               attention's workspace serves.
 * Writes nothing but the appended rows (and their per-token scales).  Two
 * sequences whose new rows coincide race; callers give distinct rows.
 */
fd_status fd_append_kv(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                       const int32_t *kv_start_idx, const int32_t *block_table,
                       int block_table_stride, const int32_t *positions, int64_t kv_rows,
                       int batch, int n_new, int num_kv_heads, int head_dim, int page_size,
                       float k_scale, float v_scale, fd_scale_kind scale_kind, float *k_scales,
                       float *v_scales, fd_dtype new_dtype, fd_dtype kv_dtype, void *workspace,
                       size_t workspace_bytes, fd_stream_t stream);

/*
 * One decode (q_len = 1) or verify (q_len > 1) step with its KV append:
 * fd_append_kv of the step's q_len new tokens (k_new, v_new
 * [batch, q_len, num_kv_heads, head_dim] of q_dtype, the first at
 * `positions`), then fd_decode_attention_multi over the caches that now hold
 * them, in one call.  seq_len counts the new tokens (typically
 * positions[b] + q_len).  The split kernel of the attention is
 * launched as a programmatic dependent of the append: its plan overlaps the
 * append, and it waits for the append's writes before reading K/V.
 * Arguments and errors are those of the two functions; nothing is launched
 * when any argument is invalid.
 */
fd_status fd_decode_attention_append(const void *q, const void *k_new, const void *v_new,
                                     void *k_cache, void *v_cache, const int32_t *kv_start_idx,
                                     const int32_t *block_table, int block_table_stride,
                                     const int32_t *positions, const int32_t *seq_len,
                                     int64_t kv_rows, int batch, int q_len, int num_q_heads,
                                     int num_kv_heads, int head_dim, int page_size,
                                     float softmax_scale, float k_scale, float v_scale,
                                     fd_scale_kind scale_kind, float *k_scales, float *v_scales,
                                     fd_dtype q_dtype, fd_dtype kv_dtype, void *out, float *lse,
                                     void *workspace, size_t workspace_bytes, fd_stream_t stream);

/*
 * Same computation as fd_decode_attention, for callers that cannot allocate
 * device memory (for example code running inside a framework that does not
 * expose its allocator, or under a fixed memory budget).  The pages have no
 * counterpart of this function; it exists only for those callers.
 *
 * Arguments are those of fd_decode_attention without the workspace: the
 * scratch memory is a 16 MiB array compiled into the library, which every
 * GPU that loads the library holds until the process exits.  Sizes whose
 * fd_workspace_bytes(...) exceeds 16 MiB return FD_ERR_WORKSPACE_TOO_SMALL
 * before any launch.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  Each call first clears the array's
 * device-error word, so device-side bounds errors of this entry point are not
 * reported; use fd_decode_attention when they must be.  All calls share the
 * one array: calls that can overlap on the GPU (different streams, or
 * different host threads) race on it and must be serialised by the caller.
 * Nothing is allocated or freed.  Invalid or unsupported arguments get the
 * same status as from fd_decode_attention.  The array's address is kept for
 * the life of the process: do not call this entry point after
 * cudaDeviceReset.
 */
fd_status fd_decode_attention_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *kv_start_idx, const int32_t *block_table,
                                      int block_table_stride, const int32_t *seq_len,
                                      int64_t kv_rows, int batch, int num_q_heads,
                                      int num_kv_heads, int head_dim, int page_size,
                                      float softmax_scale, float k_scale, float v_scale,
                                      fd_dtype q_dtype, fd_dtype kv_dtype, void *out, float *lse,
                                      fd_stream_t stream);

/*
 * Synchronises `stream`, reads and clears the workspace's sticky device-error
 * word.  Returns FD_OK, FD_ERR_DEVICE_BOUNDS, FD_ERR_DEVICE_TIMEOUT or
 * FD_ERR_CUDA.  If info is not NULL it receives the first offending value
 * (a row or page id) or 0.
 */
fd_status fd_check_device_error(void *workspace, fd_stream_t stream, int64_t *info);

/* Static English text for a status code. */
const char *fd_status_string(fd_status status);

/* Process-wide choice of the split kernel (default FD_KERNEL_AUTO). */
fd_status fd_set_kernel(fd_kernel kernel);

/*
 * Kernel that fd_decode_attention would run for these sizes under the
 * current fd_set_kernel choice: FD_KERNEL_SIMT, FD_KERNEL_MMA, FD_KERNEL_TC or FD_KERNEL_FMA,
 * or -1 if the sizes are unsupported (num_q_heads counts every query token:
 * query heads times q_len).  The answer is for per-tensor or per-KV-head
 * scales; fd_selected_kernel_scaled answers for per-token scales too.  Host
 * function.
 */
int fd_selected_kernel(int num_q_heads, int num_kv_heads, int head_dim, fd_dtype q_dtype,
                       fd_dtype kv_dtype, int paged, int page_size);

/*
 * As fd_selected_kernel, for a call with finer K/V scales of `scale_kind`
 * (FD_SCALE_TENSOR gives the same answer as fd_selected_kernel): the kernel
 * that fd_decode_attention_scaled (or _multi, _append) would run, or -1 when
 * the call would return FD_ERR_UNSUPPORTED (for instance a forced
 * FD_KERNEL_TC or FD_KERNEL_FMA with FD_SCALE_TOKEN).  Host function.
 */
int fd_selected_kernel_scaled(int num_q_heads, int num_kv_heads, int head_dim, fd_dtype q_dtype,
                              fd_dtype kv_dtype, int paged, int page_size,
                              fd_scale_kind scale_kind);

/*
 * Profiling hook: when both events are non-NULL, fd_decode_attention records
 * `before` immediately before and `after` immediately after the split
 * kernel's launch on its stream, so that the split kernel can be timed by
 * itself.  NULL, NULL switches it off.  The setting is per host thread.
 */
fd_status fd_set_split_events(fd_event_t before, fd_event_t after);

/*
 * Test hook: copies the split plan of the last fd_decode_attention call that
 * used this workspace into host memory (synchronises `stream`).
 * plan[0..7] = {num_streams, streams_per_sequence, tile_tokens, grid,
 * total_units, units_per_cta, kernel, start_units}; stream j of sequence b
 * serves query heads [j * h, (j + 1) * h) with h = num_q_heads /
 * streams_per_sequence.  A stream with n > 0 tiles costs start_units + n
 * plan units (the start cost first), an empty stream none; CTA c takes units
 * [c * units_per_cta, (c + 1) * units_per_cta).
 * plan[8 .. 8 + num_streams] = exclusive prefix of units per stream
 * (num_streams + 1 values).  capacity = number of int32 that fit in plan.
 */
fd_status fd_debug_read_plan(const void *workspace, fd_stream_t stream, int32_t *plan,
                             int capacity);

/*
 * Test hook: gathers, with the kernels' own addressing, the stored K (or V)
 * row slice of every token of every sequence into dst, a dense device array
 * [sum_b seq_len[b], num_kv_heads, head_dim] of the cache element type,
 * sequences in order.  Rows out of range are written as zero bytes and
 * recorded like in fd_decode_attention.  Same layout arguments as
 * fd_decode_attention; workspace needs only the 256-byte header.
 */
fd_status fd_debug_gather_kv(const void *cache, const int32_t *kv_start_idx,
                             const int32_t *block_table, int block_table_stride,
                             const int32_t *seq_len, int64_t kv_rows, int batch,
                             int num_kv_heads, int head_dim, int page_size, fd_dtype kv_dtype,
                             void *dst, void *workspace, fd_stream_t stream);

/*
 * Test hook for the bounded waits of the tensor-core split kernel.  Every
 * wait of that kernel on its copy pipeline gives up after `wait_ns`
 * nanoseconds (0: the default of one second), records
 * FD_ERR_DEVICE_TIMEOUT in the workspace's error word and ends the CTA's
 * work; the asynchronous-error reporting this follows is the one of
 * "SGLang Prefill optimisation: dissecting FlashAttention kernel bottlenecks
 * with GPU Trace", section 4.2 (a device error is found by a later host
 * check, not at the launch).  With `starve_first_stage` non-zero the
 * producer of every CTA issues no copy, so the consumers' first wait runs out
 * with nothing in flight: the call itself returns FD_OK, its outputs are
 * undefined, and fd_check_device_error reports FD_ERR_DEVICE_TIMEOUT.  The
 * wait that drains copies already issued before a CTA exits keeps its own
 * one-second bound and reports FD_ERR_DEVICE_TIMEOUT too when it gives up.
 * Process-wide, from the next call on; wait_ns outside [0, 1e10] is
 * FD_ERR_INVALID_ARG.  The CUDA-core split kernel has no such waits.
 */
fd_status fd_debug_set_wait_limit(int64_t wait_ns, int starve_first_stage);

/*
 * Test hook: the segments of the split plan that each CTA of the split
 * kernel takes for these sizes, computed on the device by the split kernels'
 * own plan and segment walk (the plan of "Learn CUDA from scratch, chapter
 * 15", section 15.13: ragged batches scan their real lengths).  Arguments as
 * in fd_decode_attention_multi (paged: a block table is used, page_size its
 * page size; kv_start_idx, which the plan reads ahead for the first
 * segment of every CTA, may be NULL).  dst is a device int32 array of dst_len values, of which the
 * first grid * (1 + 5 * capacity_per_cta) are written: row c holds the
 * number of segments of CTA c, then (stream, t_begin, t_end, complete, slot)
 * for each of its first capacity_per_cta segments.  *grid_out (host) always
 * receives the grid; a dst_len too small for it returns FD_ERR_INVALID_ARG
 * before any launch.  A workspace of fd_workspace_bytes for these sizes is
 * needed (its plan words are written as by a decode call).  Asynchronous on
 * `stream`.
 */
fd_status fd_debug_plan_segments(const int32_t *seq_len, const int32_t *kv_start_idx, int batch,
                                 int q_len, int num_q_heads,
                                 int num_kv_heads, int head_dim, int paged, int page_size,
                                 fd_dtype q_dtype, fd_dtype kv_dtype, int32_t *dst,
                                 int64_t dst_len, int capacity_per_cta, int *grid_out,
                                 void *workspace,
                                 size_t workspace_bytes, fd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FD_ATTENTION_H_ */
