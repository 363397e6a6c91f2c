/*
 * pgqa.h -- C ABI of libpgqa: ragged (varlen) GQA prefill and paged GQA decode on
 * GB300 (sm_103a).
 *
 * Every entry point takes plain device pointers, sizes and a CUDA stream; no C++ or
 * framework types cross this boundary and nothing is thrown.  All calls are
 * asynchronous on `stream`: they enqueue kernels and return a status code without
 * synchronising.  Argument checks that need no device data happen on the host and
 * return an error before anything is enqueued; checks of device-resident data
 * (indptr arrays, page ids) happen in the kernels, which record failures in a device
 * status word that pgqa_get_device_status() reads.
 *
 * Conventions shared by all calls
 *   - bf16 tensors are contiguous, row-major, NHD ("token, head, dim") and 16-byte
 *     aligned.  Element [t, h, c] of a [T, H, D] tensor is at ((t * H) + h) * D + c.
 *   - Query head h reads KV head h / (num_qo_heads / num_kv_heads): consecutive query
 *     heads share a KV head (grouped-query attention).
 *   - lse is the natural-log log-sum-exp of the *scaled* scores of each output row,
 *     lse = ln sum_j exp(sm_scale * q.k_j), in fp32.  A row with no visible key gets
 *     an output of exact zeros and lse = -inf.  lse may be NULL (not written).
 *   - The caller owns every tensor.  The library owns only its workspace (below).
 *   - Calls that share a workspace must be ordered (same stream, or synchronised):
 *     two in flight at once race on it.
 *
 * Sources (restated): Atlas "Module flashinfer" API page (ragged_prefill_bf16_hd128,
 * ragged_prefill_bf16_hd256: one varlen launch over q_indptr / kv_indptr, bf16, GQA,
 * causal selectable; callers pass device pointers plus a cudaStream_t);
 * vllm-rlt pull request "feat: add FlashInfer attention backend for SM120 decode"
 * (Scope and Design notes: paged NHD decode, block size 16, empty batch returns early,
 * padding in the block table is never visible, lazily allocated kernel workspace);
 * FlashInfer documentation (flashinfer_benchmark.py Attention Flags: bottom-right
 * causal masking; flashinfer.cascade "Merge Attention States": merging partial
 * (output, lse) pairs, used by the split-KV decode).
 */
#ifndef PGQA_H_
#define PGQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t / CUstream (NULL = the legacy default stream). */
typedef struct CUstream_st* pgqa_stream_t;

/* Status codes returned by every call (0 = success). */
enum {
    PGQA_OK = 0,
    PGQA_ERR_INVALID_ARG = -1,    /* NULL pointer, negative size, misaligned tensor */
    PGQA_ERR_UNSUPPORTED = -2,    /* shape outside the supported set (see each call) */
    PGQA_ERR_WORKSPACE = -3,      /* workspace too small and allocation not allowed */
    PGQA_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed */
    PGQA_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait expired (device status) */
    PGQA_ERR_DEVICE_BOUNDS = -6,  /* bad indptr / page id seen on the device */
    PGQA_ERR_NO_DEVICE = -7,      /* no usable sm_103 GPU for this call */
    PGQA_ERR_DEVICE_CAPACITY = -8 /* a prefill's work list outgrew the workspace (device
                                     status); nothing was written */
};

/*
 * Ragged (varlen) batched prefill attention in one launch.
 *
 * Defined by: Atlas "Module flashinfer" API page, functions ragged_prefill_bf16_hd128 and
 * ragged_prefill_bf16_hd256 (batched varlen prefill over q_indptr / kv_indptr offsets);
 * causal alignment from FlashInfer documentation, flashinfer_benchmark.py "Attention
 * Flags" (--causal, bottom-right masking).
 *
 *   q  [total_q, num_qo_heads, head_dim]  bf16, device     (read)
 *   k  [total_kv, num_kv_heads, head_dim] bf16, device     (read)
 *   v  [total_kv, num_kv_heads, head_dim] bf16, device     (read)
 *   o  [total_q, num_qo_heads, head_dim]  bf16, device     (written, rows of requests)
 *   lse [total_q, num_qo_heads]           fp32, device or NULL (written)
 *   q_indptr, kv_indptr [batch + 1] int32, device: request b owns query rows
 *       q_indptr[b] .. q_indptr[b+1]-1 and key rows kv_indptr[b] .. kv_indptr[b+1]-1.
 *       Both must be non-decreasing and non-negative; total_q = q_indptr[batch] and
 *       total_kv = kv_indptr[batch] are read on the device, never on the host.
 *   causal != 0: query row i of a request (0-based) sees key j iff
 *       j <= i + kv_len - qo_len  (bottom-right aligned); else every key of its request.
 *   sm_scale: scores are sm_scale * q.k (any finite value, 0 allowed).
 *
 * Split: with head_dim 128, a call whose work list would have fewer than two items per
 * SM cuts each request's keys into chunks of 2048 and merges the chunks' partial
 * results by their log-sum-exp (when the partial rows fit in the workspace).  The choice
 * is made on the device from the whole call, and the chunks of a request depend on that
 * request alone, so among calls that take the same choice a request's results do not
 * depend on the rest of the batch, bit for bit.
 *
 * Supported: head_dim 128 or 256; num_qo_heads a multiple of num_kv_heads with group
 * size G = num_qo_heads / num_kv_heads dividing 128.  batch == 0 returns PGQA_OK at once.
 * With batch > 0 every pointer but lse must be non-NULL even where total_q or total_kv is
 * 0 (the totals are never read on the host); a buffer of one row serves, since no row
 * outside the indptr ranges is read.
 * Errors: PGQA_ERR_INVALID_ARG for NULL/misaligned pointers or bad counts,
 * PGQA_ERR_UNSUPPORTED for other shapes, PGQA_ERR_WORKSPACE if the workspace is too
 * small while the stream is being captured (or a caller-supplied workspace cannot hold
 * the per-request arrays plus 4096 work items), PGQA_ERR_CUDA on a launch failure.  A
 * decreasing or negative indptr is reported later as PGQA_ERR_DEVICE_BOUNDS by
 * pgqa_get_device_status() and nothing is written.  A work list (one item per kv head and
 * pair of 128-row query tiles, or per such item and 2048-key chunk when split) longer than
 * the workspace holds is reported as PGQA_ERR_DEVICE_CAPACITY and nothing is written:
 * give the library a workspace of pgqa_workspace_bytes_prefill() bytes.  The lazily
 * allocated 128 MiB workspace holds about 690,000 items.
 */
int pgqa_ragged_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* q_indptr, const int32_t* kv_indptr, int batch,
                             int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                             float sm_scale, pgqa_stream_t stream);

/*
 * Paged prefill / append: ragged query rows over a paged NHD KV cache in one launch.  The
 * keys of request b are its cached prefix followed by the new tokens' keys, already
 * written into its pages by the caller, kv_lens[b] keys in all; its qo_len query rows are
 * the last qo_len positions (bottom-right causal alignment).  Decode of several tokens per
 * request (speculative verification) is the case of small qo_len.
 *
 * Defined by: FlashInfer documentation, flashinfer.prefill
 * (BatchPrefillWithPagedKVCacheWrapper: batched prefill / append attention of ragged
 * queries over a paged KV cache with page_size, NHD layout, causal masking aligned to the
 * bottom right, flashinfer_benchmark.py "Attention Flags"); the page-table addressing and
 * padding rules are those of the paged decode below (vllm-rlt pull request "feat: add
 * FlashInfer attention backend for SM120 decode", Design notes).
 *
 *   q  [total_q, num_qo_heads, head_dim] bf16, device (read); rows of request b are
 *       q_indptr[b] .. q_indptr[b+1]-1 (q_indptr [batch + 1] int32, device, as for
 *       pgqa_ragged_prefill_bf16; total_q = q_indptr[batch] is read on the device)
 *   k_pages, v_pages [num_pages, page_size, num_kv_heads, head_dim] bf16, device (read)
 *   page_table [batch, page_table_stride] int32, device: key j of request b is slot
 *       j % page_size of page page_table[b * page_table_stride + j / page_size]; entries at
 *       index >= ceil(kv_lens[b] / page_size) are never read.
 *   kv_lens [batch] int32, device: 0 <= kv_lens[b] <= page_table_stride * page_size.
 *   o [total_q, num_qo_heads, head_dim] bf16, lse [total_q, num_qo_heads] fp32 or NULL:
 *       written for every query row, as for pgqa_ragged_prefill_bf16.
 *   causal != 0: query row i (0-based within its request) sees key j iff
 *       j <= i + kv_len - qo_len; else every key of its request.
 *   Key slots past kv_lens[b] in a request's last page are never used, so whatever they
 *   hold (even NaN) cannot reach the output.
 *   Split-KV for short work lists (a few requests with few query rows over long keys) as
 *   for pgqa_ragged_prefill_bf16.
 *
 * Supported: head_dim 128 or 256; page_size 16, 32, 64 or 128; G = num_qo_heads /
 * num_kv_heads dividing 128.  batch == 0 returns PGQA_OK at once.  Errors as for
 * pgqa_ragged_prefill_bf16 (including PGQA_ERR_DEVICE_CAPACITY for a work list longer
 * than the workspace holds); a kv_len outside its range or a decreasing q_indptr is
 * reported as PGQA_ERR_DEVICE_BOUNDS by pgqa_get_device_status() and nothing is written;
 * a page id outside 0..num_pages-1 is reported the same way and that page is not read
 * (the rows that need it are then undefined).
 */
int pgqa_paged_prefill_bf16(const void* q, const void* k_pages, const void* v_pages, void* o,
                            float* lse, const int32_t* q_indptr, const int32_t* page_table,
                            int page_table_stride, const int32_t* kv_lens, int page_size,
                            int num_pages, int batch, int num_qo_heads, int num_kv_heads,
                            int head_dim, int causal, float sm_scale, pgqa_stream_t stream);

/*
 * Paged decode: one query row per request over a paged NHD KV cache, split along the
 * keys (split-KV) with the partial results merged by log-sum-exp weights.
 *
 * Defined by: vllm-rlt pull request "feat: add FlashInfer attention backend for SM120
 * decode" (Scope: paged decode; Design notes: block tables with -1 / zero / stale
 * padding stay invisible, kv_layout "NHD", empty batch returns early) and FlashInfer
 * documentation, flashinfer.decode (BatchDecodeWithPagedKVCacheWrapper) and
 * flashinfer.cascade "Merge Attention States" (the split-KV merge).
 *
 *   q       [batch, num_qo_heads, head_dim]                 bf16, device (read)
 *   k_pages [num_pages, page_size, num_kv_heads, head_dim]  bf16, device (read)
 *   v_pages [num_pages, page_size, num_kv_heads, head_dim]  bf16, device (read)
 *   page_table [batch, page_table_stride] int32, device: key j of request b is slot
 *       j % page_size of page page_table[b * page_table_stride + j / page_size].
 *       Entries at index >= ceil(kv_lens[b] / page_size) are never read.
 *   kv_lens [batch] int32, device: 0 <= kv_lens[b] <= page_table_stride * page_size.
 *   o   [batch, num_qo_heads, head_dim] bf16, device (written)
 *   lse [batch, num_qo_heads] fp32, device or NULL (written)
 *   Key slots past kv_lens[b] in a request's last page are never read, so whatever
 *   they hold (even NaN) cannot reach the output.
 *
 * Split: each request's keys are cut into chunks of C keys, C the longest of 1024, 512,
 * 256, 128 for which batch * ceil(page_table_stride * page_size / C) * num_kv_heads >= 2048
 * (128 if none is), a choice made from these sizes alone.  For a given C a request's
 * result does not depend on the other requests of the batch, bit for bit.
 *
 * Supported: head_dim 128; page_size 16, 32, 64 or 128; G = num_qo_heads / num_kv_heads in
 * {1,2,4,8}.
 * Errors as for pgqa_ragged_prefill_bf16; a page id outside 0..num_pages-1 or a
 * kv_len outside its range is reported as PGQA_ERR_DEVICE_BOUNDS by
 * pgqa_get_device_status(), and the affected request's keys are skipped.
 */
int pgqa_paged_decode_bf16(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, const int32_t* kv_lens, int page_size,
                           int page_table_stride, int num_pages, void* o, float* lse,
                           int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                           float sm_scale, pgqa_stream_t stream);

/*
 * The paged prefill and the paged decode over K/V pools of any layout whose head_dim
 * elements are contiguous: element [page, slot, head, c] of k_pages (and v_pages, which
 * must have the same layout) is at
 *     page * page_stride + slot * slot_stride + head * head_stride + c      (elements).
 * Covers the packed NHD layout of the calls above (page_stride = page_size * Hk * d,
 * slot_stride = Hk * d, head_stride = d), the HND layout [num_pages, Hk, page_size, d]
 * (page_stride = Hk * page_size * d, slot_stride = d, head_stride = page_size * d), and a
 * per-layer slice of a larger cache such as [num_pages, num_layers, page_size, Hk, d]
 * (page_stride = num_layers * page_size * Hk * d, others as for NHD).
 *
 * Defined by: the calls above (same arguments, results and supported shapes); the NHD /
 * HND kv_layout choice is FlashInfer documentation, flashinfer_benchmark.py "Attention
 * Flags" (--kv_layout), and non-contiguous per-layer slices of the cache are inputs the
 * vllm-rlt pull request "feat: add FlashInfer attention backend for SM120 decode" tests
 * its decode kernel on (its GPU test suite: oracle parity on non-contiguous layer slices).
 *
 * Strides are in elements: positive multiples of 8 (16 bytes) and below 2^36, else
 * PGQA_ERR_INVALID_ARG.  k_pages / v_pages must be 16-byte aligned.
 */
int pgqa_paged_prefill_bf16_strided(const void* q, const void* k_pages, const void* v_pages,
                                    void* o, float* lse, const int32_t* q_indptr,
                                    const int32_t* page_table, int page_table_stride,
                                    const int32_t* kv_lens, int page_size, int num_pages,
                                    int64_t page_stride, int64_t slot_stride, int64_t head_stride,
                                    int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                                    int causal, float sm_scale, pgqa_stream_t stream);
int pgqa_paged_decode_bf16_strided(const void* q, const void* k_pages, const void* v_pages,
                                   const int32_t* page_table, const int32_t* kv_lens,
                                   int page_size, int page_table_stride, int num_pages,
                                   int64_t page_stride, int64_t slot_stride, int64_t head_stride,
                                   void* o, float* lse, int batch, int num_qo_heads,
                                   int num_kv_heads, int head_dim, float sm_scale,
                                   pgqa_stream_t stream);

/*
 * Paged decode over an FP8 E4M3 KV cache: k_pages / v_pages hold one byte per element
 * (OCP E4M3, "fn": no infinities, S.1111.111 is NaN) and the element values are
 * e4m3 * k_scale (keys) and e4m3 * v_scale (values), one scale per tensor.  q, o and lse
 * stay bf16 / bf16 / fp32; everything else is as for pgqa_paged_decode_bf16_strided, with
 * strides in elements (= bytes) that must be positive multiples of 16.  For packed NHD
 * pools pass page_stride = page_size * Hk * d, slot_stride = Hk * d, head_stride = d.
 *
 * Defined by: FlashInfer documentation, flashinfer_benchmark.py "Attention Flags"
 * (--kv_dtype fp8_e4m3: E4M3 key and value tensors); the pages give no scale convention,
 * so one float scale per tensor is taken (flashinfer "FP8 GEMM: Per-tensor and groupwise
 * scaling" lists per-tensor scaling as one of its FP8 modes).
 *
 * Arithmetic: the products run on the tensor cores with E4M3 operands; q (scaled by a power
 * of two) and the softmax weights enter as sums of two E4M3 values (q exactly down to about
 * 2^-9 of its largest element, the weights to about 8 significant bits, as a bf16 P), with
 * fp32 accumulation.  Results are within the tolerance of the other entry points.
 *
 * Supported: head_dim 128; page_size 16, 32, 64 or 128; G in {1,2,4,8}.  Errors as for
 * pgqa_paged_decode_bf16; a NaN or infinite scale is PGQA_ERR_INVALID_ARG.
 */
int pgqa_paged_decode_e4m3(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, const int32_t* kv_lens, int page_size,
                           int page_table_stride, int num_pages, int64_t page_stride,
                           int64_t slot_stride, int64_t head_stride, float k_scale, float v_scale,
                           void* o, float* lse, int batch, int num_qo_heads, int num_kv_heads,
                           int head_dim, float sm_scale, pgqa_stream_t stream);

/*
 * Paged prefill over an FP8 E4M3 KV cache: the computation of pgqa_paged_prefill_bf16 with
 * K/V stored as in pgqa_paged_decode_e4m3 (one byte per element, values e4m3 * k_scale and
 * e4m3 * v_scale, strides in elements = bytes, positive multiples of 16).
 *
 * Defined by: FlashInfer documentation, flashinfer.prefill
 * (BatchPrefillWithPagedKVCacheWrapper: ragged queries over a paged KV cache, causal
 * masking aligned to the bottom right) with flashinfer_benchmark.py "Attention Flags"
 * (--kv_dtype fp8_e4m3 for the prefill and decode routines); scale convention as for
 * pgqa_paged_decode_e4m3.
 *
 *   q [total_q, num_qo_heads, head_dim] bf16 and q_indptr [batch + 1] int32 (device) as
 *       for pgqa_paged_prefill_bf16.
 *   max_qo_len: the most query rows any request has (q_indptr stays on the device); it
 *       chooses the path below.
 *   page_table, kv_lens, page_size, num_pages: as for pgqa_paged_prefill_bf16.
 *   o [total_q, num_qo_heads, head_dim] bf16, lse [total_q, num_qo_heads] fp32 or NULL.
 *   causal != 0: query row i of a request with qo_len rows and kv_len keys sees key j iff
 *       j <= i + kv_len - qo_len (a row that sees no key gets zeros and lse = -inf).
 *
 * Two paths, the same results up to rounding:
 *   - head_dim 128, G in {1,2,4,8} and max_qo_len * G <= 16 (multi-token decode,
 *     speculative verification): the tensor-core E4M3 decode, each request's query rows
 *     as the columns of its MMAs, so the keys stream once for all of them; split-KV as for
 *     the decode, with chunks of at most 896 keys when max_qo_len > 1.  A request with
 *     more than max_qo_len rows is reported as PGQA_ERR_DEVICE_BOUNDS and none of its rows
 *     is written.
 *   - otherwise: the pages the call reads are converted into the workspace, K to bf16 and
 *     V to f16 (both exact), then the paged prefill runs over them with k_scale folded into
 *     the score scale, v_scale into the output scale and the weights P rounded to f16 for
 *     P.V (at least the accuracy of the bf16 paged prefill over the same values).  The
 *     conversion needs 2 * P * page_size * num_kv_heads * head_dim * 2 bytes of workspace
 *     on top of the prefill's own, P = min(num_pages, batch * page_table_stride); a
 *     caller workspace too small for it gives PGQA_ERR_WORKSPACE.
 *
 * Supported: head_dim 128 or 256; page_size 16, 32, 64 or 128; G = num_qo_heads /
 * num_kv_heads dividing 128.  max_qo_len < 1 (with batch > 0), a NULL q_indptr or a NaN /
 * infinite scale is PGQA_ERR_INVALID_ARG.  Other errors as for pgqa_paged_prefill_bf16; a
 * page id outside 0..num_pages-1 is reported as PGQA_ERR_DEVICE_BOUNDS and that page is
 * not read (the rows that need it are then undefined).
 */
int pgqa_paged_prefill_e4m3(const void* q, const void* k_pages, const void* v_pages, void* o,
                            float* lse, const int32_t* q_indptr, const int32_t* page_table,
                            int page_table_stride, const int32_t* kv_lens, int page_size,
                            int num_pages, int64_t page_stride, int64_t slot_stride,
                            int64_t head_stride, float k_scale, float v_scale, int batch,
                            int max_qo_len, int num_qo_heads, int num_kv_heads, int head_dim,
                            int causal, float sm_scale, pgqa_stream_t stream);

/* Same calls under the short names used by serving integrations. */
int ragged_prefill_bf16(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* q_indptr, const int32_t* kv_indptr, int batch,
                        int num_qo_heads, int num_kv_heads, int head_dim, int causal,
                        float sm_scale, pgqa_stream_t stream);
int paged_prefill_bf16(const void* q, const void* k_pages, const void* v_pages, void* o,
                       float* lse, const int32_t* q_indptr, const int32_t* page_table,
                       int page_table_stride, const int32_t* kv_lens, int page_size,
                       int num_pages, int batch, int num_qo_heads, int num_kv_heads,
                       int head_dim, int causal, float sm_scale, pgqa_stream_t stream);
int paged_decode_bf16(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* page_table, const int32_t* kv_lens, int page_size,
                      int page_table_stride, int num_pages, void* o, float* lse, int batch,
                      int num_qo_heads, int num_kv_heads, int head_dim, float sm_scale,
                      pgqa_stream_t stream);

/*
 * Paged decode that allocates nothing.  The source pages have no counterpart for this
 * call: it is an addition of this library.
 *
 * Same arguments, results and supported shapes as pgqa_paged_decode_bf16.  That call keeps
 * its split-KV partial results in a workspace it cudaMalloc's on first use (and grows when
 * a call needs more).  Some callers cannot let a library allocate device memory: serving
 * engines that hand all free device memory to their own pool (KV cache, activations) at
 * start-up, so a later cudaMalloc fails or fragments that pool; and deployments that
 * forbid allocation once initialisation is over (real-time or certified systems, where
 * every byte is budgeted up front).  This call keeps its scratch in a fixed 16 MiB array
 * in the library's own static device memory instead, which every GPU that loads the
 * library holds until the process exits.  The caller still passes (and owns) every input
 * and output.
 *
 *   - Set-up: the first call on each device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and keeps it.
 *   - Limit: returns PGQA_ERR_WORKSPACE, enqueueing nothing, when
 *       1024 + 256-rounded (2*batch+1)*4 + 256-rounded C*Hq*4 + C*Hq*head_dim*4 > 16 MiB,
 *     with C = batch * ceil(page_table_stride * page_size / K) partial chunks and K the
 *     chunk length chosen as for pgqa_paged_decode_bf16 (e.g. batch 16 with 32k-key
 *     tables at 32 query heads fits; batch 32 does not).
 *   - Sharing: every call on a device uses the same array and leaves its contents
 *     behind (each call clears what it needs cleared); calls that overlap on the GPU
 *     (different streams without ordering) race and corrupt each other's results.  Order
 *     them.
 *   - Device-side errors are not reported: pgqa_get_device_status() does not see this
 *     call's status word.  Bad page ids and kv_lens are handled as in
 *     pgqa_paged_decode_bf16 (the bad keys are skipped).  If a bounded wait expires (the
 *     2 s device timeout), the warp gives up and the rows it was working on hold
 *     undefined values; the call still returned PGQA_OK.
 * No cudaMalloc, cudaFree or other allocating call is made.
 */
int pgqa_paged_decode_bf16_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                   const int32_t* page_table, const int32_t* kv_lens,
                                   int page_size, int page_table_stride, int num_pages,
                                   void* o, float* lse, int batch, int num_qo_heads,
                                   int num_kv_heads, int head_dim, float sm_scale,
                                   pgqa_stream_t stream);

/*
 * Workspace.  Every call needs device scratch: the prefills for their work list and
 * tensor maps, the decode for its split-KV partial results.  Unless the caller supplies one,
 * the library allocates it lazily on the first call that needs it (per device; 128 MiB
 * or more if the call needs more) and grows it when a call needs more -- except while
 * `stream` is being captured into a CUDA graph, where it returns PGQA_ERR_WORKSPACE
 * instead of allocating (run one call before capturing, as with the pages' lazily
 * allocated 128 MiB workspace: vllm-rlt PR, Design notes).
 *
 * pgqa_set_workspace: use caller-owned device memory `ptr` of `bytes` bytes (256-byte
 *   aligned) on the current device from now on; the library frees its own buffer.
 *   ptr == NULL drops a caller buffer and returns to lazy allocation.  The buffer must
 *   stay valid until replaced and must not be used by anything else meanwhile.
 * pgqa_workspace_bytes_*: upper bound of the bytes a call with these sizes needs.
 *   For the prefills (ragged and paged), max_total_q bounds q_indptr[batch].
 */
int pgqa_set_workspace(void* ptr, size_t bytes);
size_t pgqa_workspace_bytes_prefill(int batch, int64_t max_total_q, int num_qo_heads,
                                    int num_kv_heads);
size_t pgqa_workspace_bytes_decode(int batch, int page_table_stride, int page_size,
                                   int num_qo_heads, int head_dim);

/*
 * Device status: synchronises `stream`, returns the first error the kernels recorded on
 * the current device since the last call (PGQA_OK, PGQA_ERR_DEVICE_TIMEOUT,
 * PGQA_ERR_DEVICE_BOUNDS) and clears it.  Returns PGQA_ERR_CUDA if the stream itself
 * reports an error.
 */
int pgqa_get_device_status(pgqa_stream_t stream);

/*
 * Self-test of the device-side failure path.  Enqueues on `stream` one warp that waits,
 * with the same bounded mbarrier wait as every kernel of this library, on a barrier that
 * nothing arrives at.  After the wait limit (2 s) the kernel records PGQA_DEV_TIMEOUT in
 * this device's status word, plus where it gave up, and returns; the next
 * pgqa_get_device_status() reports PGQA_ERR_DEVICE_TIMEOUT and clears both.  Nothing
 * else is touched, and the context stays usable.  Creates the workspace if there is
 * none.  Returns PGQA_OK once enqueued, or PGQA_ERR_NO_DEVICE / PGQA_ERR_CUDA.
 */
int pgqa_selftest_expired_wait(pgqa_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* pgqa_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int pgqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PGQA_H_ */
