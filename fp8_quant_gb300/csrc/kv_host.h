// Host-side helpers shared by the KV-cache entry points: CUDA error capture,
// per-device SM counts, occupancy, the launch wrapper (programmatic
// dependent launch, one warp per unit) and argument/alignment helpers.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "kv_device.cuh"

namespace kvimpl {

extern thread_local int g_last_cuda_error;

kv_status cuda_fail(cudaError_t e);

// Where the input buffers live.  Inputs may be device memory or page-locked
// host memory the device reads directly (NVLink-C2C / PCIe); memory unknown to
// CUDA is rejected with KV_ERR_INVALID_ARG.  *all_device is true when every
// input is device (or managed-free device-resident) memory, which is when the
// kernels may prefetch inputs into L2 with bulk copies.
kv_status classify_inputs(const void* const* ptrs, int n, bool* all_device);

// The fused dynamic per-tensor write's state (kv_store_fp8_dynamic_tensor):
// work = {generation, tagged K maximum, tagged V maximum}, each tagged word
// (generation << 16) | the 16-bit pattern of max |x|; scale_out receives the
// forward scales amax / fmax.
struct DynTensor {
  uint64_t* work;
  float* scale_out[2];
  float fmax;
};

// The FP8 write with a per-tensor inverse scale (or none), or one inverse
// scale per page of scale_page slots (scale_page > 0), in format fmt
// (kFmtE4M3 / kFmtE5M2): kv_store_fp8 and the static modes of kv_store_fp8_ex.
// dyn non-null: the inverse scales come from the tagged maxima instead (the
// fused dynamic per-tensor write; inv pointers unused, use_scale 1).
kv_status store_fp8_static(const void* k, const void* v, void* k_cache, void* v_cache,
                           const void* indices, kv_index_dtype index_dtype, int64_t index_stride,
                           int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                           kv_src_dtype src_dtype, const kv_strides* s, int64_t page_size,
                           int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                           const float* inv_k_scale, const float* inv_v_scale, int32_t use_scale,
                           int64_t scale_page, int fmt, kv_error_record* d_err,
                           kv_stream_t stream, const DynTensor* dyn = nullptr);

// The absmax reduction (kv_scale.cu) into acc (two 32-bit float-bit
// accumulators) or, when tagged is non-null, into the fused write's tagged
// workspace.  The callers check the arguments; num_tokens > 0.
kv_status absmax_reduce(const void* k, const void* v, kv_src_dtype src_dtype, int64_t num_tokens,
                        int32_t num_heads, int32_t head_dim, const kv_strides* s,
                        unsigned int* acc, uint64_t* tagged, bool on_device, cudaStream_t stream);
kv_status current_sm_count(int* out);
kv_status blocks_per_sm(const void* fn, int threads, int* out);

// Threads per CTA of a launch over num_units warps of work.  Small launches
// are latency-bound and prefer fewer, larger CTAs; large launches stream
// better with smaller CTAs (measured on GB300).
inline int launch_threads(uint64_t num_units) {
  return num_units >= KV_LARGE_LAUNCH_WARPS ? KV_THREADS_LARGE : KV_THREADS;
}

// Grid: enough CTAs for every unit to have a warp, capped at the resident
// capacity (a whole number of CTAs per SM) and at max_ctas; warps loop over
// the rest.  threads_override > 0 fixes the CTA size.
template <typename Params>
kv_status launch(void (*kernel)(Params), uint64_t num_units, const Params& params,
                 cudaStream_t stream, uint64_t max_ctas = 0, int threads_override = 0) {
  const int threads = threads_override > 0 ? threads_override : launch_threads(num_units);
  const uint64_t warps = static_cast<uint64_t>(threads / 32);
  int sms = 0, per_sm = 0;
  kv_status st = current_sm_count(&sms);
  if (st != KV_OK) return st;
  st = blocks_per_sm(reinterpret_cast<const void*>(kernel), threads, &per_sm);
  if (st != KV_OK) return st;
  const uint64_t want = (num_units + warps - 1) / warps;
  // One warp per unit lets the CTA scheduler balance the load across SMs
  // (a fixed per-warp share of units was measured ~10% slower on large
  // batches); the loop in the kernels covers grids beyond the dimension limit.
  const uint64_t cap = KV_GRID_WAVES > 0
                           ? static_cast<uint64_t>(sms) * static_cast<uint64_t>(per_sm) * KV_GRID_WAVES
                           : uint64_t{0x7FFFFFFF};
  uint64_t grid64 = want < cap ? want : cap;
  if (max_ctas != 0 && grid64 > max_ctas) grid64 = max_ctas;
  if (grid64 == 0) grid64 = 1;
  const unsigned grid = static_cast<unsigned>(grid64);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, params);
  if (e != cudaSuccess) return cuda_fail(e);
  return KV_OK;
}

// launch() for the row gathers and the dynamic-scale write, which prefetch
// ahead: when the launch runs in more than one wave of resident CTAs and
// moves at most KV_LOOKAHEAD_MAX_BYTES (launch_bytes: read + written),
// params.ahead is set to the resident warps, and each warp prefetches into L2
// what the warp that will take its place one wave later is going to read.
// In a gather that hides the slot -> row dependency of the later waves
// (gather_fp8 8.84 -> 8.65 us), and in the dynamic write the row's arrival
// before its scale can be formed (fp8_dynamic 9.58 -> 9.2 us).  A launch
// whose traffic exceeds L2 by far loses more to prefetched rows evicted
// before use than it gains (gather_prefill, 268 MB: 39.2 us without, 41.2
// with).  The static writes, whose row loads do not wait on the slot,
// measured slower with it (fp8 7.68 -> 7.88 us, strided 78.6 -> 81.6 us) and
// do not use it.
template <typename Params>
kv_status launch_rows(void (*kernel)(Params), uint64_t num_units, Params params,
                      cudaStream_t stream, uint64_t launch_bytes) {
  params.ahead = 0;
  if (KV_LOOKAHEAD && params.prefetch && launch_bytes <= KV_LOOKAHEAD_MAX_BYTES) {
    const int threads = launch_threads(num_units);
    int sms = 0, per_sm = 0;
    kv_status st = current_sm_count(&sms);
    if (st != KV_OK) return st;
    st = blocks_per_sm(reinterpret_cast<const void*>(kernel), threads, &per_sm);
    if (st != KV_OK) return st;
    const uint64_t resident = static_cast<uint64_t>(sms) * static_cast<uint64_t>(per_sm) *
                              static_cast<uint64_t>(threads / 32);
    if (num_units > resident) params.ahead = resident;
  }
  return launch(kernel, num_units, params, stream);
}

// Largest power of two <= KV_MAX_VEC dividing every value OR-ed into `bits`.
inline int pow2_align(uint64_t bits) {
  int v = KV_MAX_VEC;
  while (v > 1 && (bits & static_cast<uint64_t>(v - 1)) != 0) v >>= 1;
  return v;
}

inline uint64_t u64(const void* p) { return static_cast<uint64_t>(reinterpret_cast<uintptr_t>(p)); }
inline uint64_t u64(int64_t x) { return static_cast<uint64_t>(x); }

inline bool common_args_ok(const void* k, const void* v, const void* k_cache, const void* v_cache,
                    const void* indices, kv_index_dtype index_dtype, int64_t index_stride,
                    int32_t num_heads, int32_t head_dim, const kv_strides* s, int64_t size_limit,
                    const kv_error_record* d_err) {
  if (!k || !v || !k_cache || !v_cache || !indices || !s || !d_err) return false;
  if (index_dtype != KV_INDEX_I32 && index_dtype != KV_INDEX_I64) return false;
  if (index_stride < 1 || num_heads < 1 || head_dim < 1 || size_limit < 0) return false;
  if ((u64(d_err) & 7u) != 0) return false;
  return true;
}

// Segments: one per row when heads are contiguous on every side, else one
// per head.
struct Segments {
  uint32_t count;
  int64_t elems;  // elements per segment
};

inline Segments segments(int32_t num_heads, int32_t head_dim, int64_t src_head_bytes,
                  int64_t dst_head_bytes, const kv_strides* s) {
  if (num_heads == 1 ||
      (s->k_head == src_head_bytes && s->v_head == src_head_bytes &&
       s->kc_head == dst_head_bytes && s->vc_head == dst_head_bytes))
    return Segments{1u, static_cast<int64_t>(num_heads) * head_dim};
  return Segments{static_cast<uint32_t>(num_heads), static_cast<int64_t>(head_dim)};
}

// Automatic split: small batches get more warps per row so that the copy
// spreads over every SM; a part keeps at least one chunk per lane.
inline uint32_t auto_parts(uint64_t units, int64_t seg_chunks, int sms) {
  uint32_t parts = 1;
  while (units * parts < static_cast<uint64_t>(sms) * 16u && seg_chunks % (2 * parts) == 0 &&
         seg_chunks / (2 * parts) >= 32 && parts < 8)
    parts *= 2;
  return parts;
}

}  // namespace kvimpl
