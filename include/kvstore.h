/*
 * kvstore.h -- C ABI of the GB300 (sm_103a) KV-cache write library.
 *
 * For every new token t, the K row and the V row (num_heads x head_dim
 * elements, arbitrary byte strides) are written into row indices[t] of a
 * large K cache and V cache:
 *
 *   kv_store      plain byte-exact copy of the rows;
 *   kv_store_fp8  each element is widened to fp32, optionally multiplied by a
 *                 per-tensor fp32 inverse scale, converted to FP8 e4m3fn and
 *                 written at the paged cache address of the slot.
 *
 * Sources (sglang): kvcache.cuh, kernel `store_kvcache` and host launcher
 * `StoreKVCacheKernel::run` (plain copy, the row-split option and the slot
 * bound 0 <= slot < size_limit); trtllm_fp8_kv_kernel.py, kernels
 * `_fused_fp8_set_kv_buffer_kernel` / `_process_kv_tensor` and the wrapper
 * `fused_fp8_set_kv_buffer` (page decomposition, strides, fp32 inverse scale
 * read on the device, e4m3fn conversion).
 *
 * Conventions shared by every call:
 *  - All tensor pointers are memory owned by the caller; the library never
 *    allocates, frees or retains them, and never allocates memory of its own
 *    during a call.  Caches and error records are device memory
 *    (kv_error_snapshot may also write to page-locked host memory).  The
 *    token-major side of every call -- the inputs of the writes (k, v) and
 *    the outputs of the gathers (k_out, v_out) -- and the slot ids may also
 *    be page-locked host memory (cudaHostAlloc / cudaHostRegister), which the
 *    kernels read or write in place over NVLink-C2C or PCIe.  Pointers CUDA
 *    does not know (pageable host memory, stray addresses) are rejected with
 *    KV_ERR_INVALID_ARG before anything is launched.
 *  - Calls are asynchronous on `stream` and do not synchronise the host,
 *    except kv_error_poll.  They may be captured in a CUDA graph.
 *  - Every kernel launched here waits for the work that precedes it on the
 *    stream before it touches memory (programmatic dependent launch), so the
 *    stream's ordering is kept.
 *  - Strides are in BYTES and may be any int64 value; elements of one head
 *    are contiguous when the dim stride equals the element size, which is the
 *    fast path.  Bases and strides that are not 16-byte multiples select
 *    narrower vector widths; this is never an error.
 *  - An out-of-range slot (outside [0, size_limit)) is not an argument error:
 *    the kernel skips that token (neither its K nor its V row is written),
 *    counts it in the caller's error record and continues.  kv_error_poll
 *    reports it.  No slot value can cause a write outside the rows
 *    [0, size_limit) of the caches.
 *  - size_limit is trusted to be at most the number of cache rows.
 *  - Duplicate slots: calls write the candidate rows concurrently, so each
 *    element of such a cache row equals the same element of one of the
 *    candidate rows; which candidate is unspecified and may differ from
 *    element to element (and between the K and the V row).
 *  - The inputs and the index array must not overlap the caches.
 *  - num_tokens == 0 returns KV_OK without launching (pointers may be NULL).
 */
#ifndef FP8_QUANT_GB300_KVSTORE_H
#define FP8_QUANT_GB300_KVSTORE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KV_ABI_VERSION 1

/* Same type as cudaStream_t.  NULL selects the legacy default stream. */
typedef struct CUstream_st *kv_stream_t;

typedef enum kv_status {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,  /* bad argument found on the host; nothing was launched */
    KV_ERR_UNSUPPORTED = 2,  /* legal request this library does not implement; nothing launched */
    KV_ERR_CUDA = 3,         /* a CUDA runtime call failed; see kv_last_cuda_error() */
    KV_ERR_INDEX_OOB = 4     /* kv_error_poll: at least one token had an out-of-range slot */
} kv_status;

typedef enum kv_index_dtype { KV_INDEX_I32 = 0, KV_INDEX_I64 = 1 } kv_index_dtype;

/* Element type of the K/V inputs of kv_store_fp8 (2-byte floats). */
typedef enum kv_src_dtype { KV_SRC_F16 = 0, KV_SRC_BF16 = 1 } kv_src_dtype;

/* Byte strides.  Element (t, h, d) of K is at k + t*k_token + h*k_head +
 * d*k_dim; element (h, d) of cache row s is at k_cache + s*kc_slot +
 * h*kc_head + d*kc_dim (kv_store_fp8 adds the page decomposition, below).
 * The K cache and the V cache have separate strides. */
typedef struct kv_strides {
    int64_t k_token, k_head, k_dim;
    int64_t v_token, v_head, v_dim;
    int64_t kc_slot, kc_head, kc_dim;
    int64_t vc_slot, vc_head, vc_dim;
} kv_strides;

/* Device-side error record, owned by the caller (16 bytes, 8-byte aligned,
 * zero-initialised before first use, e.g. with cudaMemsetAsync or
 * kv_error_reset).  Kernels only add to it; kv_error_poll reads and clears it.
 * Calls that share one record on different streams share its counts. */
typedef struct kv_error_record {
    uint64_t oob_count;      /* tokens skipped because their slot was out of range */
    uint64_t first_bad_key;  /* bitwise NOT of the lowest skipped token; 0 if none */
} kv_error_record;

/*
 * kv_store -- plain copy (sglang kvcache.cuh, `store_kvcache`).
 *
 *   k, v           device pointers to element (0, 0, 0) of the K and V inputs.
 *   k_cache,
 *   v_cache        device pointers to element (slot 0, 0, 0) of the caches.
 *   indices        device pointer to num_tokens slot ids (int32 or int64 per
 *                  index_dtype), read at indices[t * index_stride]
 *                  (index_stride in ELEMENTS, >= 1).
 *   num_heads,
 *   head_dim       row shape, both >= 1.
 *   elem_bytes     element size: 1, 2, 4 or 8 (the copy is byte-exact, so the
 *                  element type does not matter; bf16/fp16 rows use 2).
 *   strides        byte strides (host pointer, read during the call only).
 *   size_limit     slots must satisfy 0 <= slot < size_limit.
 *   num_split      how many parts each contiguous row is split into, each
 *                  part copied by its own warp: 0 = choose automatically,
 *                  1, 2 or 4.  2 and 4 need the row's bytes (num_heads *
 *                  head_dim * elem_bytes) to be a multiple of 256 and 512
 *                  respectively (the split rule of `StoreKVCacheKernel`);
 *                  otherwise KV_ERR_INVALID_ARG.  The result does not depend
 *                  on num_split.
 *   d_err          device error record (required when num_tokens > 0).
 *   stream         CUDA stream.
 *
 * Returns KV_OK once the kernel is enqueued, KV_ERR_INVALID_ARG for a bad
 * argument (NULL pointer, num_tokens < 0, num_heads/head_dim < 1, bad
 * elem_bytes, index_dtype, index_stride, num_split or split rule, size_limit
 * < 0, misaligned d_err), KV_ERR_CUDA if the launch failed.
 */
kv_status kv_store(const void *k, const void *v, void *k_cache, void *v_cache,
                   const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                   int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                   int32_t elem_bytes, const kv_strides *strides, int64_t size_limit,
                   int32_t num_split, kv_error_record *d_err, kv_stream_t stream);

/*
 * kv_store_paged -- kv_store into a paged cache [pages, page_size, H, D]
 * whose page stride may include padding: slot s is written at
 * (s / page_size) * kc_page_stride + (s % page_size) * kc_slot + h * kc_head
 * + d * kc_dim (likewise for V), the 4-D write of trtllm_fp8_kv_kernel.py
 * `_naive_fp8_set_kv_buffer` (k_cache[page_ids, page_offsets] = k) for a
 * cache of the input's own type.  A page stride of page_size * kc_slot is
 * the flat layout of kv_store.  Other arguments and errors as kv_store, plus
 * KV_ERR_INVALID_ARG for page_size < 1.
 */
kv_status kv_store_paged(const void *k, const void *v, void *k_cache, void *v_cache,
                         const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                         int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                         int32_t elem_bytes, const kv_strides *strides, int64_t page_size,
                         int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                         int32_t num_split, kv_error_record *d_err, kv_stream_t stream);

/*
 * kv_store_fp8 -- fused scale + FP8 e4m3fn conversion + paged write
 * (sglang trtllm_fp8_kv_kernel.py, `_fused_fp8_set_kv_buffer_kernel`,
 * `_process_kv_tensor`, wrapper `fused_fp8_set_kv_buffer`).
 *
 * Arguments as for kv_store, except:
 *   k, v           bf16 or fp16 inputs (src_dtype); addresses and the
 *                  k/v strides must be even.
 *   k_cache,
 *   v_cache        caches of e4m3fn bytes (kc_dim / vc_dim are the byte
 *                  distance between consecutive dims, normally 1).
 *   page_size      tokens per page, >= 1.  Slot s is written at
 *                  (s / page_size) * kc_page_stride + (s % page_size) * kc_slot
 *                  + h * kc_head + d * kc_dim (likewise for V).  A 3-D cache
 *                  [slots, H, D] passes kc_page_stride = page_size * kc_slot,
 *                  which makes this s * kc_slot; a 4-D cache
 *                  [pages, page_size, H, D] passes its page stride.
 *   inv_k_scale,
 *   inv_v_scale    DEVICE pointers to one fp32 each (the inverse scales),
 *                  read by the kernel, so no host synchronisation is needed;
 *                  both must be non-NULL when use_scale != 0 and are ignored
 *                  otherwise.
 *   use_scale      0: convert x unscaled; else convert fl32(x * inv).
 *
 * Numerics (per element): x is widened exactly to fp32; y = x * inv in fp32
 * with round-to-nearest-even (no fused operations, denormals kept); the code
 * is the e4m3fn value nearest to y, ties to the even mantissa, with finite
 * overflow and +-Inf saturated to +-448 and every NaN written as 0x7F.
 * use_scale == 0 gives the same bytes as use_scale != 0 with inv = 1.0f.
 *
 * Returns as kv_store; KV_ERR_INVALID_ARG also for a bad src_dtype,
 * page_size < 1, odd input addresses or strides, or a NULL scale pointer
 * with use_scale != 0.
 */
kv_status kv_store_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                       const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                       int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                       kv_src_dtype src_dtype, const kv_strides *strides, int64_t page_size,
                       int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                       const float *inv_k_scale, const float *inv_v_scale, int32_t use_scale,
                       kv_error_record *d_err, kv_stream_t stream);

/*
 * kv_gather -- the inverse of kv_store: row t of k_out / v_out takes the cache
 * row of slot indices[t], byte for byte.  The single-GPU counterpart of the
 * materialise step of vLLM dcp_direct_kv_gather.cu
 * (`materialize_kv_gather_kernel`), and the read-back half of a round trip.
 *
 * Arguments as for kv_store with the roles of the tensors swapped: k_cache /
 * v_cache are read, k_out / v_out are written.  In `strides`, k_* / v_*
 * describe the OUTPUT rows and kc_* / vc_* the caches.  An out-of-range slot
 * leaves output row t untouched and is counted in d_err.  The outputs must
 * not overlap the caches or the indices.
 */
kv_status kv_gather(const void *k_cache, const void *v_cache, void *k_out, void *v_out,
                    const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                    int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                    int32_t elem_bytes, const kv_strides *strides, int64_t size_limit,
                    kv_error_record *d_err, kv_stream_t stream);

/*
 * kv_gather_paged -- kv_gather from a paged cache [pages, page_size, H, D]
 * (the inverse of kv_store_paged): slot s is read at
 * (s / page_size) * kc_page_stride + (s % page_size) * kc_slot + ... .
 * Other arguments and errors as kv_gather, plus KV_ERR_INVALID_ARG for
 * page_size < 1.
 */
kv_status kv_gather_paged(const void *k_cache, const void *v_cache, void *k_out, void *v_out,
                          const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                          int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                          int32_t elem_bytes, const kv_strides *strides, int64_t page_size,
                          int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                          kv_error_record *d_err, kv_stream_t stream);

/*
 * kv_gather_fp8 -- dequantising gather from e4m3fn caches written by
 * kv_store_fp8 (same page addressing: page_size, kc_page_stride,
 * vc_page_stride).  Each code is decoded exactly to fp32, multiplied by the
 * fp32 scale (k_scale / v_scale: DEVICE pointers, the forward scales, i.e.
 * 1/inv) when use_scale != 0, and rounded to nearest-even bf16 or fp16
 * (out_dtype).  NaN codes become the canonical NaN 0x7FFF; fp16 overflow
 * becomes +-Inf.  Output strides (k_* / v_*) must be even.
 */
kv_status kv_gather_fp8(const void *k_cache, const void *v_cache, void *k_out, void *v_out,
                        const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                        int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                        kv_src_dtype out_dtype, const kv_strides *strides, int64_t page_size,
                        int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                        const float *k_scale, const float *v_scale, int32_t use_scale,
                        kv_error_record *d_err, kv_stream_t stream);

/* FP8 cache formats of the extended calls. */
typedef enum kv_fp8_format {
    KV_FP8_E4M3FN = 0,   /* largest finite 448, no infinities */
    KV_FP8_E5M2 = 1      /* largest finite 57344 */
} kv_fp8_format;

/* Scale modes of the extended calls. */
typedef enum kv_scale_mode {
    KV_SCALE_NONE = 0,        /* values converted unscaled */
    KV_SCALE_TENSOR = 1,      /* one fp32 scale per tensor, a device scalar */
    KV_SCALE_TOKEN = 2,       /* one scale per token row (all heads), computed per call */
    KV_SCALE_TOKEN_HEAD = 3,  /* one scale per (token, head), computed per call */
    KV_SCALE_PAGE = 4         /* one fp32 scale per cache page, supplied by the caller */
} kv_scale_mode;

/*
 * kv_store_fp8_ex -- kv_store_fp8 with a choice of FP8 format and of scale
 * granularity, including scales computed in the kernel.  The fused FP8
 * write's module docstring (trtllm_fp8_kv_kernel.py) names per-token scale
 * computation and e5m2 caches; its kernel implements the per-tensor e4m3fn
 * case only, which is kv_store_fp8 (= this call with KV_FP8_E4M3FN and
 * KV_SCALE_TENSOR or KV_SCALE_NONE).
 *
 * Arguments as kv_store_fp8, plus:
 *   format       KV_FP8_E4M3FN or KV_FP8_E5M2 (rounding: nearest even; finite
 *                overflow and infinities saturate to the largest finite
 *                value; every NaN becomes 0x7F).
 *   scale_mode   KV_SCALE_NONE / KV_SCALE_TENSOR: as kv_store_fp8 with
 *                use_scale 0 / 1 (inv_k_scale, inv_v_scale are device
 *                pointers to the inverse scales).
 *                KV_SCALE_TOKEN / KV_SCALE_TOKEN_HEAD: for each group (the
 *                token's K row or V row, or one head of it) the kernel takes
 *                amax = max |x| (NaN ignored), inv = fmax / amax and
 *                scale = amax / fmax in fp32 round-to-nearest (both 1 when
 *                amax is 0; fmax = 448 or 57344), writes the codes of
 *                fl32(x * inv), and stores `scale` (the dequantisation
 *                multiplier) at k_scales[slot * scales_slot_stride + g],
 *                g = head (TOKEN_HEAD) or 0 (TOKEN); likewise V.  The scale
 *                caches are device float arrays indexed by slot, not by page.
 *                KV_SCALE_PAGE: inv_k_scale / inv_v_scale point to device
 *                arrays of fp32 INVERSE scales, one per cache page; the
 *                token written to slot s uses inv[s / page_size] in place of
 *                the per-tensor scalar (codes of fl32(x * inv[s / page_size])).
 *                The arrays must hold ceil(size_limit / page_size) floats.
 *                The fused FP8 write's module docstring names per-page scales
 *                and its kernel has none; the page is the one its kernel
 *                computes, slot // page_size.  Any layout kv_store_fp8 takes.
 *   k_scales,
 *   v_scales,
 *   scales_slot_stride   used by the dynamic modes only: non-NULL, 4-byte
 *                aligned, stride >= num_heads (TOKEN_HEAD) or >= 1 (TOKEN).
 * The dynamic modes need contiguous dims (k_dim = v_dim = 2, kc_dim = vc_dim
 * = 1), else KV_ERR_UNSUPPORTED.  Out-of-range slots write neither codes nor
 * scales.
 */
kv_status kv_store_fp8_ex(const void *k, const void *v, void *k_cache, void *v_cache,
                          const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                          int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                          kv_src_dtype src_dtype, const kv_strides *strides, int64_t page_size,
                          int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                          kv_fp8_format format, kv_scale_mode scale_mode,
                          const float *inv_k_scale, const float *inv_v_scale, float *k_scales,
                          float *v_scales, int64_t scales_slot_stride, kv_error_record *d_err,
                          kv_stream_t stream);

/*
 * kv_gather_fp8_ex -- kv_gather_fp8 for every layout kv_store_fp8_ex writes:
 * codes of `format` decoded exactly, multiplied by the scale of `scale_mode`
 * (NONE: none; TENSOR: *k_scale / *v_scale, the forward scales; TOKEN /
 * TOKEN_HEAD: k_scales[slot * scales_slot_stride + g] as written by
 * kv_store_fp8_ex; PAGE: k_scale[slot / page_size] / v_scale[...], device
 * arrays of forward scales, one per cache page), rounded to bf16 / fp16.
 * kv_gather_fp8 is this call with KV_FP8_E4M3FN and NONE / TENSOR.
 */
kv_status kv_gather_fp8_ex(const void *k_cache, const void *v_cache, void *k_out, void *v_out,
                           const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                           int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                           kv_src_dtype out_dtype, const kv_strides *strides, int64_t page_size,
                           int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                           kv_fp8_format format, kv_scale_mode scale_mode, const float *k_scale,
                           const float *v_scale, const float *k_scales, const float *v_scales,
                           int64_t scales_slot_stride, kv_error_record *d_err,
                           kv_stream_t stream);

/*
 * kv_inv_scale -- inv[i] = 1 / scale[i] in fp32, round to nearest, for
 * i < n, on the device (trtllm_fp8_kv_kernel.py, `fused_fp8_set_kv_buffer`
 * forms 1.0 / k_scale on the GPU so that graph capture needs no host sync).
 * scale and inv are device pointers to n floats (4-byte aligned; they may be
 * the same array).  n == 0: KV_OK, nothing launched.
 */
kv_status kv_inv_scale(const float *scale, float *inv, int64_t n, kv_stream_t stream);

/*
 * kv_absmax_inv -- per-tensor scale of the K rows and of the V rows on the
 * device: amax[0] = max |K|, amax[1] = max |V| over all num_tokens x num_heads
 * x head_dim elements (NaN elements ignored; 0 for an empty or all-NaN
 * tensor), and inv[j] = fp8_max / amax[j] in fp32 round-to-nearest (1.0 when
 * amax[j] is 0).  With fp8_max = 448 this is the per-tensor inverse scale
 * kv_store_fp8 takes (e4m3fn's largest finite value maps to the tensor's
 * largest magnitude).
 *   k, v       bf16 / fp16 rows (src_dtype); strides->k_* and v_* are used
 *              (dims must be contiguous: k_dim = v_dim = 2; else
 *              KV_ERR_UNSUPPORTED).
 *   amax, inv  device pointers to two floats each, written by the call.
 *   work       NULL, or a device workspace of KV_ABSMAX_WORK_BYTES (4-byte
 *              aligned) owned by the caller: zero before its first use (e.g.
 *              cudaMemsetAsync), and left zero by every call that completes.
 *              With it a call is two kernels (reduce, finish); without it,
 *              three (amax is cleared by a kernel first and serves as the
 *              accumulator).  Calls that share one workspace must not
 *              overlap on the GPU (their maxima would mix); calls on one
 *              stream never do.
 * fp8_max must be positive and finite.
 */
#define KV_ABSMAX_WORK_BYTES 8
kv_status kv_absmax_inv(const void *k, const void *v, kv_src_dtype src_dtype,
                        int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                        const kv_strides *strides, float fp8_max, float *amax, float *inv,
                        uint32_t *work, kv_stream_t stream);

/*
 * kv_store_fp8_dynamic_tensor -- the FP8 write with per-tensor scales formed
 * from the batch itself, in one call: the fused form of kv_absmax_inv
 * followed by kv_store_fp8_ex in KV_SCALE_TENSOR mode (the trtllm page's
 * docstring advertises computed scales while its kernel takes a given one;
 * the recipe is the per-tensor one, inv = fmax / amax).
 *   amax_k = max |K| and amax_v = max |V| over all num_tokens rows (NaN
 *   elements ignored; out-of-range slots do not exclude their rows), then
 *   inv = fmax / amax in fp32 round-to-nearest (1.0 when amax is 0) and the
 *   codes fp8(fl32(x * inv)) as kv_store_fp8_ex writes them; fmax is 448
 *   (e4m3fn) or 57344 (e5m2).  *k_scale / *v_scale receive the forward
 *   (dequantisation) scales amax / fmax (1.0 when amax is 0), what
 *   kv_gather_fp8_ex takes in KV_SCALE_TENSOR mode.
 * Arguments as kv_store_fp8_ex, plus:
 *   k_scale, v_scale  device pointers to one float each (4-byte aligned).
 *   work   device workspace of KV_DYNAMIC_TENSOR_WORK_BYTES (8-byte aligned),
 *          owned by the caller, zero before its first use.  It holds a
 *          generation counter and the two maxima tagged with it, so a call
 *          needs no clearing pass: two kernels (the reduction, then the
 *          write, which forms the inverse scales in its prologue).  Calls
 *          sharing one workspace must not overlap on the GPU; calls on one
 *          stream never do.  After a KV_ERR_CUDA return its contents are
 *          undefined: zero it again before the next call.
 * Dims must be contiguous on the input side (k_dim = v_dim = 2; else
 * KV_ERR_UNSUPPORTED); the cache side may use any layout kv_store_fp8_ex
 * takes.  num_tokens == 0: KV_OK, nothing launched, nothing written.
 */
#define KV_DYNAMIC_TENSOR_WORK_BYTES 24
kv_status kv_store_fp8_dynamic_tensor(const void *k, const void *v, void *k_cache,
                                      void *v_cache, const void *indices,
                                      kv_index_dtype index_dtype, int64_t index_stride,
                                      int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                                      kv_src_dtype src_dtype, const kv_strides *strides,
                                      int64_t page_size, int64_t kc_page_stride,
                                      int64_t vc_page_stride, int64_t size_limit,
                                      kv_fp8_format format, float *k_scale, float *v_scale,
                                      uint64_t *work, kv_error_record *d_err, kv_stream_t stream);

/*
 * kv_store_noalloc -- kv_store for callers that cannot allocate device memory.
 * The pages have no counterpart; this entry point exists for this library's
 * users only.
 *
 * Some callers cannot call cudaMalloc at the point where they write the KV
 * cache: code running inside an allocator hook (where allocating would
 * re-enter the allocator), a plugin that is handed the tensors but owns no
 * memory pool, or a process whose device memory is entirely reserved by a pool
 * it does not control.  kv_store needs one more device buffer besides the
 * tensors, its error record, so those callers could not use it.
 * kv_store_noalloc takes the same arguments as kv_store except d_err and
 * allocates nothing: the record lives in a 256-byte static device array inside
 * this library (KV_NOALLOC_SCRATCH_BYTES), which every GPU that loads the
 * library holds until the process exits.  The record needs 16 bytes whatever
 * the batch size, so no batch exceeds the array; a build whose record did not
 * fit would return KV_ERR_UNSUPPORTED.
 *
 * Behaviour:
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress); make that first call
 *    before any stream capture on the device.  The address is kept with the
 *    id of the CUDA context it was found in; a call from another context (for
 *    instance after cudaDeviceReset) looks it up again.
 *  - Each call clears the record on `stream`, runs kv_store with it, then
 *    synchronises `stream` and copies the record to *oob_count and
 *    *first_bad_token (host, nullable; -1 when no token was skipped).  It
 *    therefore blocks the host until the write has finished.
 *  - It makes CUDA API calls, so it must not be called from a stream callback
 *    or a host function enqueued with cudaLaunchHostFunc, where CUDA forbids
 *    them.
 *  - Every call shares the one array: calls that overlap on the GPU (from
 *    other host threads or on other streams) race on it and may report each
 *    other's counts.  The cache writes themselves are not affected.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Returns KV_OK, KV_ERR_INDEX_OOB when a token was skipped, or the status of
 * kv_store / of a failed CUDA call.
 */
#define KV_NOALLOC_SCRATCH_BYTES 256
kv_status kv_store_noalloc(const void *k, const void *v, void *k_cache, void *v_cache,
                           const void *indices, kv_index_dtype index_dtype, int64_t index_stride,
                           int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                           int32_t elem_bytes, const kv_strides *strides, int64_t size_limit,
                           int32_t num_split, int64_t *oob_count, int64_t *first_bad_token,
                           kv_stream_t stream);

/*
 * kv_error_poll -- synchronise `stream`, read the error record, clear it.
 * (The pages trap inside the kernel on a bad slot; this library reports it
 * here instead.)  Writes the number of skipped tokens and the lowest skipped
 * token (-1 if none) to the optional host outputs.  Returns KV_OK when no
 * token was skipped, KV_ERR_INDEX_OOB when one was, KV_ERR_INVALID_ARG for a
 * NULL or misaligned record, KV_ERR_CUDA if a CUDA call failed (including an
 * earlier asynchronous error surfaced by the synchronisation).
 * Not capturable in a CUDA graph (it synchronises).
 */
kv_status kv_error_poll(kv_error_record *d_err, kv_stream_t stream, int64_t *oob_count,
                        int64_t *first_bad_token);

/* kv_error_snapshot -- copy the record to `dst` asynchronously on `stream`,
 * as it stands once the work before it on the stream has finished.  A small
 * kernel (capturable, chained by programmatic launch), so a captured step can
 * hand its status to the host without a copy-engine transfer: `dst` may be
 * device memory or page-locked host memory (read it after synchronising).
 * The record is not cleared.  Both pointers 8-byte aligned; memory unknown to
 * CUDA is rejected with KV_ERR_INVALID_ARG. */
kv_status kv_error_snapshot(const kv_error_record *d_err, kv_error_record *dst,
                            kv_stream_t stream);

/* kv_error_reset -- zero the record asynchronously on `stream` (capturable). */
kv_status kv_error_reset(kv_error_record *d_err, kv_stream_t stream);

/* kv_launch_floor -- a measurement aid with no counterpart on the pages.
 * Launches an empty kernel sized for num_warps warps of work, with the CTA
 * size, grid and programmatic-launch attributes the write kernels use for
 * that much work, and the same wait for the preceding grid.  It touches no
 * memory.  Timed back to back on a stream, it gives the fixed cost that every
 * launch of this library pays, the floor under a small call such as a decode
 * step (256 tokens of 2048-byte rows run as 1,024 warps).  num_warps in
 * [1, 2^40], else KV_ERR_INVALID_ARG. */
kv_status kv_launch_floor(int64_t num_warps, kv_stream_t stream);

/* Static, NUL-terminated name of a status code. */
const char *kv_status_str(kv_status status);

/* The cudaError_t value of the last failed CUDA call made by this library on
 * the calling thread (0 if none). */
int kv_last_cuda_error(void);

/* KV_ABI_VERSION of the library that was loaded. */
int kv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8_QUANT_GB300_KVSTORE_H */
