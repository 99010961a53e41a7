// KV-cache write kernels for GB300 (sm_103a) and the C ABI declared in
// include/kvstore.h.
//
// What is computed (sglang kvcache.cuh, `store_kvcache`; sglang
// trtllm_fp8_kv_kernel.py, `_fused_fp8_set_kv_buffer_kernel` and
// `_process_kv_tensor`): for each token t with slot s = indices[t], the K row
// and the V row are written into cache row s -- byte for byte (kv_store) or
// as FP8 e4m3fn after an fp32 multiply by the inverse scale (kv_store_fp8).
//
// Design.  The path is a pure HBM stream (no arithmetic worth a tensor core),
// so every choice is about bytes in flight and coalescing:
//  * A row is cut into "segments" (one per head, or one per row when heads
//    are contiguous on both sides) and optionally into parts; a unit of work
//    is (token, K|V, segment, part) and one warp moves one unit at a time.
//  * Lane l of the warp moves chunks l, l+32, l+64, ... of the unit, so every
//    warp-wide load or store covers 32 consecutive chunks (512 contiguous
//    bytes at 16 B per chunk): full 32-byte sectors, one request per 4 lines.
//  * The unit's first batch of loads (up to U chunks per lane) is issued
//    before the slot id is known, so the index read and the row read overlap;
//    only the stores depend on the slot.
//  * Loads are non-coherent and do not allocate in L1 (the rows are read
//    once); the grid is a whole number of CTAs per SM and loops over units.
//  * Out-of-range slots are skipped and counted in the caller's error record
//    with two atomics per bad token; nothing traps and nothing is written
//    outside [0, size_limit).
//  * Every kernel waits on the previous grid (griddepcontrol.wait) before its
//    first global access and is launched with programmatic stream
//    serialisation, so its launch overlaps the previous kernel's tail.
#include <cuda.h>  // context types of the driver entry points fetched at run time

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "kv_host.h"

#ifndef KV_STORE_PAIR
#define KV_STORE_PAIR 1   // large FP8 writes: one warp moves the K and the V part of a token
#endif

namespace kvimpl {

thread_local int g_last_cuda_error = 0;

// ---------------------------------------------------------------------------
// Plain copy: kvcache.cuh `store_kvcache` / `copy_kv_warp`.
// ---------------------------------------------------------------------------

struct CopySide {
  const uint8_t* src;  // element (0, 0, 0) of the input
  uint8_t* dst;        // element (slot 0, 0, 0) of the cache
  int64_t src_token, src_seg, dst_slot, dst_seg;
  int64_t dst_page;    // page stride (the slot stride when page_size == 1)
};

struct CopyParams {
  CopySide side[2];
  const void* indices;
  int64_t index_stride;
  int64_t size_limit;
  int64_t page_size;  // 1: flat cache (slot * slot stride)
  UnitShape shape;
  kv_error_record* err;
  int prefetch;  // sources are 16-byte aligned: prefetch them into L2 before the grid wait
  int vec;       // bytes per chunk (the kernel's VEC / OUT)
};

// Moves one unit: loads (issued before the slot is known), bounds check,
// stores.  `src` already points at the unit's first source byte.
template <int VEC, int U, typename IdxT>
__device__ __forceinline__ void copy_unit(const CopyParams& p, const Unit& w, const uint8_t* src,
                                          uint32_t lane) {
  const uint32_t nchunks = p.shape.part_chunks;
  const int64_t part_bytes = static_cast<int64_t>(nchunks) * VEC;
  const CopySide& sd = p.side[w.kv];
  const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, w.token);
  Chunk<VEC> buf[U];
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const uint32_t c = lane + 32u * j;
    if (c < nchunks) ld_stream(buf[j], src + static_cast<size_t>(c) * VEC);
  }
  if (slot < 0 || slot >= p.size_limit) {
    if (w.rank == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(w.token));
    return;
  }
  uint8_t* dst = sd.dst + paged_offset(slot, p.page_size, sd.dst_page, sd.dst_slot) +
                 static_cast<int64_t>(w.seg) * sd.dst_seg + static_cast<int64_t>(w.part) * part_bytes;
#pragma unroll
  for (int j = 0; j < U; ++j) {
    const uint32_t c = lane + 32u * j;
    if (c < nchunks) st_stream(dst + static_cast<size_t>(c) * VEC, buf[j]);
  }
  // Rows longer than 32*U chunks: further batches, loads then stores.
  for (uint32_t c0 = 32u * U; c0 < nchunks; c0 += 32u * U) {
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t c = c0 + lane + 32u * j;
      if (c < nchunks) ld_stream(buf[j], src + static_cast<size_t>(c) * VEC);
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t c = c0 + lane + 32u * j;
      if (c < nchunks) st_stream(dst + static_cast<size_t>(c) * VEC, buf[j]);
    }
  }
}

__device__ __forceinline__ const uint8_t* copy_src(const CopyParams& p, const Unit& w) {
  const CopySide& sd = p.side[w.kv];
  return sd.src + w.token * sd.src_token + static_cast<int64_t>(w.seg) * sd.src_seg +
         static_cast<int64_t>(w.part) * p.shape.part_chunks * static_cast<int64_t>(p.vec);
}

template <int VEC, int U, typename IdxT>
__global__ void __launch_bounds__(kThreads) kv_copy_rows(const __grid_constant__ CopyParams p) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
  const bool active = u < p.shape.num_units;

  // Everything that needs no memory written by the previous grid happens
  // before the wait: the first unit's coordinates and addresses, and an L2
  // prefetch of its source bytes and slot id.
  Unit w = decode_unit(p.shape, active ? u : 0);
  const uint8_t* src = copy_src(p, w);
  if (KV_PREFETCH && p.prefetch && lane == 0 && active) {
    prefetch_l2_bulk(src, p.shape.part_chunks * static_cast<uint32_t>(VEC));
    prefetch_l2_line(static_cast<const IdxT*>(p.indices) + w.token * p.index_stride);
  }
  grid_handover();

  while (u < p.shape.num_units) {
    copy_unit<VEC, U, IdxT>(p, w, src, lane);
    u += nwarps;
    if (u >= p.shape.num_units) break;
    w = decode_unit(p.shape, u);
    src = copy_src(p, w);
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// Element-wise copy for rows whose elements are not contiguous (dim stride
// different from the element size).  One warp per (token, K|V, head).
struct GenericCopyParams {
  const uint8_t* src[2];
  uint8_t* dst[2];
  int64_t src_token[2], src_head[2], src_dim[2];
  int64_t dst_slot[2], dst_head[2], dst_dim[2], dst_page[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size;
  uint64_t num_units;  // num_tokens * 2 * num_heads
  int32_t num_heads, head_dim, elem_bytes;
  kv_error_record* err;
};

template <typename IdxT>
__global__ void __launch_bounds__(kThreads) kv_copy_elements(const __grid_constant__ GenericCopyParams p) {
  grid_handover();
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  const uint64_t per_token = 2ull * static_cast<uint64_t>(p.num_heads);
  for (uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
       u < p.num_units; u += nwarps) {
    const int64_t t = static_cast<int64_t>(u / per_token);
    const uint32_t r = static_cast<uint32_t>(u - static_cast<uint64_t>(t) * per_token);
    const int kv = r >= static_cast<uint32_t>(p.num_heads) ? 1 : 0;
    const int64_t h = r - kv * p.num_heads;
    const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, t);
    if (slot < 0 || slot >= p.size_limit) {
      if (r == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(t));
      continue;
    }
    const uint8_t* src = p.src[kv] + t * p.src_token[kv] + h * p.src_head[kv];
    uint8_t* dst = p.dst[kv] + paged_offset(slot, p.page_size, p.dst_page[kv], p.dst_slot[kv]) +
                   h * p.dst_head[kv];
    for (int64_t d = lane; d < p.head_dim; d += 32) {
      const uint8_t* s = src + d * p.src_dim[kv];
      uint8_t* o = dst + d * p.dst_dim[kv];
      for (int b = 0; b < p.elem_bytes; ++b) o[b] = __ldg(s + b);
    }
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// ---------------------------------------------------------------------------
// Fused FP8 write: trtllm_fp8_kv_kernel.py `_fused_fp8_set_kv_buffer_kernel`
// and `_process_kv_tensor`.
// ---------------------------------------------------------------------------

template <int OUT> struct Fp8Chunk { uint32_t in[OUT / 2]; };

template <int OUT>
__device__ __forceinline__ void ld_in(Fp8Chunk<OUT>& c, const uint8_t* p) {
  if constexpr (OUT == 32) {
    ld_stream(*reinterpret_cast<Chunk<32>*>(&c.in[0]), p);
    ld_stream(*reinterpret_cast<Chunk<32>*>(&c.in[8]), p + 32);
  } else if constexpr (OUT == 16) {
    if constexpr (KV_MAX_VEC >= 32) {
      ld_stream(*reinterpret_cast<Chunk<32>*>(&c.in[0]), p);
    } else {
      ld_stream(*reinterpret_cast<Chunk<16>*>(&c.in[0]), p);
      ld_stream(*reinterpret_cast<Chunk<16>*>(&c.in[4]), p + 16);
    }
  } else if constexpr (OUT == 8) {
    ld_stream(*reinterpret_cast<Chunk<16>*>(&c.in[0]), p);
  } else if constexpr (OUT == 4) {
    ld_stream(*reinterpret_cast<Chunk<8>*>(&c.in[0]), p);
  } else {
    static_assert(OUT == 2, "OUT");
    ld_stream(*reinterpret_cast<Chunk<4>*>(&c.in[0]), p);
  }
}

template <int OUT, bool kBF16, int FMT>
__device__ __forceinline__ void quant_store(uint8_t* p, const Fp8Chunk<OUT>& c, float inv) {
  if constexpr (OUT >= 4) {
    Chunk<OUT> o;
#pragma unroll
    for (int i = 0; i < OUT / 4; ++i)
      o.w[i] = quant2<kBF16, FMT>(c.in[2 * i], inv) | (quant2<kBF16, FMT>(c.in[2 * i + 1], inv) << 16);
    st_stream(p, o);
  } else {
    Chunk<2> o;
    o.h = static_cast<uint16_t>(quant2<kBF16, FMT>(c.in[0], inv));
    st_stream(p, o);
  }
}

struct Fp8Side {
  const uint8_t* src;
  uint8_t* dst;
  int64_t src_token, src_seg;      // input byte strides
  int64_t dst_slot, dst_seg, dst_page;
  const float* inv;                // device scalar, or nullptr (scale 1)
};

struct Fp8Params {
  Fp8Side side[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size;
  int64_t scale_page;  // 0: side.inv is one scalar; > 0: one inverse scale per page of this size
  int scale_page_shift;  // log2(scale_page) when it is a power of two, else -1
  UnitShape shape;
  kv_error_record* err;
  int prefetch;  // sources are 16-byte aligned: prefetch them into L2 before the grid wait
  int vec;       // bytes per chunk (the kernel's VEC / OUT)
  DynTensor dyn; // dyn.work non-null: the fused dynamic per-tensor write
};

// The fused dynamic per-tensor write, after the grid wait: both sides'
// inverse scales fmax / amax from the tagged maxima the reduction left in
// the workspace (1 when amax is 0).  One thread of the grid also writes the
// forward scales amax / fmax and moves the workspace to the next generation;
// the other threads read only the tagged words, which that store leaves alone.
template <bool kBF16>
__device__ __forceinline__ void dyn_tensor_inv(const DynTensor& d, float* inv) {
  float amax[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t bits = static_cast<uint32_t>(d.work[1 + i]) & 0xFFFFu;
    amax[i] = kBF16 ? __uint_as_float(bits << 16)
                    : __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
    inv[i] = amax[i] > 0.0f ? __fdiv_rn(d.fmax, amax[i]) : 1.0f;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) d.scale_out[i][0] = amax[i] > 0.0f ? __fdiv_rn(amax[i], d.fmax) : 1.0f;
    d.work[0] = d.work[0] + 1u;
  }
}


__device__ __forceinline__ const uint8_t* fp8_src(const Fp8Params& p, const Fp8Side& sd, const Unit& w) {
  return sd.src + w.token * sd.src_token + static_cast<int64_t>(w.seg) * sd.src_seg +
         static_cast<int64_t>(w.part) * p.shape.part_chunks * 2 * static_cast<int64_t>(p.vec);
}

// One unit: loads (issued before the slot is known), bounds check, scale,
// conversion and stores.  NS == 2 moves the K and the V part of the unit
// (one slot load for both, twice the bytes in flight per warp), NS == 1 the
// side w.kv.  kDyn: the inverse scales are dyn_inv (K, V), from the fused
// dynamic per-tensor write's prologue.
template <int OUT, int U, int NS, typename IdxT, bool kBF16, int FMT, bool kDyn = false>
__device__ __forceinline__ void fp8_unit(const Fp8Params& p, const Unit& w, uint32_t lane,
                                         const float* dyn_inv = nullptr) {
  const uint32_t nchunks = p.shape.part_chunks;
  const int64_t part_out = static_cast<int64_t>(nchunks) * OUT;  // bytes out per part
  const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, w.token);
  const uint8_t* src[NS];
  float inv[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const Fp8Side& sd = p.side[NS == 2 ? i : w.kv];
    src[i] = fp8_src(p, sd, w);
    if constexpr (kDyn) inv[i] = (NS == 2 ? i : static_cast<int>(w.kv)) != 0 ? dyn_inv[1] : dyn_inv[0];
    else inv[i] = sd.inv != nullptr && p.scale_page == 0 ? __ldg(sd.inv) : 1.0f;
  }
  Fp8Chunk<OUT> buf[NS][U];
#pragma unroll
  for (int i = 0; i < NS; ++i)
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t c = lane + 32u * j;
      if (c < nchunks) ld_in<OUT>(buf[i][j], src[i] + static_cast<size_t>(c) * (2 * OUT));
    }
  if (slot < 0 || slot >= p.size_limit) {
    if (w.rank == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(w.token));
    return;
  }
  if (p.scale_page != 0) {  // per-page inverse scales: the slot's page picks the scale
    const int64_t page = p.scale_page_shift >= 0 ? slot >> p.scale_page_shift : slot / p.scale_page;
#pragma unroll
    for (int i = 0; i < NS; ++i) inv[i] = __ldg(p.side[NS == 2 ? i : w.kv].inv + page);
  }
  uint8_t* dst[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const Fp8Side& sd = p.side[NS == 2 ? i : w.kv];
    dst[i] = sd.dst + paged_offset(slot, p.page_size, sd.dst_page, sd.dst_slot) +
             static_cast<int64_t>(w.seg) * sd.dst_seg + static_cast<int64_t>(w.part) * part_out;
  }
#pragma unroll
  for (int i = 0; i < NS; ++i)
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const uint32_t c = lane + 32u * j;
      if (c < nchunks) quant_store<OUT, kBF16, FMT>(dst[i] + static_cast<size_t>(c) * OUT, buf[i][j], inv[i]);
    }
  for (uint32_t c0 = 32u * U; c0 < nchunks; c0 += 32u * U) {
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + lane + 32u * j;
        if (c < nchunks) ld_in<OUT>(buf[i][j], src[i] + static_cast<size_t>(c) * (2 * OUT));
      }
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + lane + 32u * j;
        if (c < nchunks) quant_store<OUT, kBF16, FMT>(dst[i] + static_cast<size_t>(c) * OUT, buf[i][j], inv[i]);
      }
  }
}

template <int OUT, int U, int NS, typename IdxT, bool kBF16, int FMT, bool kDyn>
__global__ void __launch_bounds__(kThreads) kv_fp8_rows(const __grid_constant__ Fp8Params p) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
  const bool active = u < p.shape.num_units;

  Unit w = decode_unit(p.shape, active ? u : 0);
  if (KV_PREFETCH && p.prefetch && lane == 0 && active) {
#pragma unroll
    for (int i = 0; i < NS; ++i)
      prefetch_l2_bulk(fp8_src(p, p.side[NS == 2 ? i : w.kv], w),
                       p.shape.part_chunks * 2u * static_cast<uint32_t>(OUT));
    prefetch_l2_line(static_cast<const IdxT*>(p.indices) + w.token * p.index_stride);
  }
  grid_handover();

  float dyn_inv[2] = {1.0f, 1.0f};
  if constexpr (kDyn) dyn_tensor_inv<kBF16>(p.dyn, dyn_inv);
  while (u < p.shape.num_units) {
    fp8_unit<OUT, U, NS, IdxT, kBF16, FMT, kDyn>(p, w, lane, dyn_inv);
    u += nwarps;
    if (u >= p.shape.num_units) break;
    w = decode_unit(p.shape, u);
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// Element-wise FP8 write for strided dims or odd sizes.  One warp per
// (token, K|V, head); lanes over the head's elements.
struct GenericFp8Params {
  const uint8_t* src[2];
  uint8_t* dst[2];
  int64_t src_token[2], src_head[2], src_dim[2];
  int64_t dst_slot[2], dst_head[2], dst_dim[2], dst_page[2];
  const float* inv[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size;
  int64_t scale_page;  // as Fp8Params::scale_page
  uint64_t num_units;
  int32_t num_heads, head_dim;
  kv_error_record* err;
  DynTensor dyn;       // as Fp8Params::dyn
};

template <typename IdxT, bool kBF16, int FMT>
__global__ void __launch_bounds__(kThreads) kv_fp8_elements(const __grid_constant__ GenericFp8Params p) {
  grid_handover();
  float dyn_inv[2] = {1.0f, 1.0f};
  if (p.dyn.work != nullptr) dyn_tensor_inv<kBF16>(p.dyn, dyn_inv);
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  const uint64_t per_token = 2ull * static_cast<uint64_t>(p.num_heads);
  for (uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
       u < p.num_units; u += nwarps) {
    const int64_t t = static_cast<int64_t>(u / per_token);
    const uint32_t r = static_cast<uint32_t>(u - static_cast<uint64_t>(t) * per_token);
    const int kv = r >= static_cast<uint32_t>(p.num_heads) ? 1 : 0;
    const int64_t h = r - kv * p.num_heads;
    const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, t);
    if (slot < 0 || slot >= p.size_limit) {
      if (r == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(t));
      continue;
    }
    const float inv = p.dyn.work != nullptr ? (kv != 0 ? dyn_inv[1] : dyn_inv[0])
                      : p.inv[kv] == nullptr ? 1.0f
                      : p.scale_page != 0 ? __ldg(p.inv[kv] + slot / p.scale_page)
                                          : __ldg(p.inv[kv]);
    const uint8_t* src = p.src[kv] + t * p.src_token[kv] + h * p.src_head[kv];
    uint8_t* dst = p.dst[kv] + paged_offset(slot, p.page_size, p.dst_page[kv], p.dst_slot[kv]) +
                   h * p.dst_head[kv];
    for (int64_t d = lane; d < p.head_dim; d += 32) {
      const uint32_t bits = __ldg(reinterpret_cast<const unsigned short*>(src + d * p.src_dim[kv]));
      dst[d * p.dst_dim[kv]] = static_cast<uint8_t>(quant2<kBF16, FMT>(bits, inv) & 0xFFu);
    }
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

kv_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return KV_ERR_CUDA;
}

kv_status classify_inputs(const void* const* ptrs, int n, bool* all_device) {
  *all_device = true;
  for (int i = 0; i < n; ++i) {
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, ptrs[i]);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();  // the query's own error is not sticky: clear it
      return cuda_fail(e);
    }
    if (a.type == cudaMemoryTypeUnregistered) return KV_ERR_INVALID_ARG;
    if (a.type != cudaMemoryTypeDevice) *all_device = false;
  }
  return KV_OK;
}

// SM count of the current device, cached per device.
std::atomic<int> g_sm_count[kMaxDevices];

kv_status current_sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < kMaxDevices) {
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) {
      *out = n;
      return KV_OK;
    }
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  *out = n;
  return KV_OK;
}

// Resident CTAs per SM of a kernel, cached per kernel (the answer is the same
// on every device this library is built for).
std::mutex g_occ_mutex;
struct OccEntry {
  const void* fn;
  int threads;
  int blocks;
};
OccEntry g_occ[256];
int g_occ_n = 0;

kv_status blocks_per_sm(const void* fn, int threads, int* out) {
  {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (int i = 0; i < g_occ_n; ++i)
      if (g_occ[i].fn == fn && g_occ[i].threads == threads) {
        *out = g_occ[i].blocks;
        return KV_OK;
      }
  }
  int b = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, 0);
  if (e != cudaSuccess) return cuda_fail(e);
  if (b < 1) b = 1;
  std::lock_guard<std::mutex> lock(g_occ_mutex);
  if (g_occ_n < 256) g_occ[g_occ_n++] = OccEntry{fn, threads, b};
  *out = b;
  return KV_OK;
}

template <int VEC, typename IdxT>
kv_status launch_copy_vec(const CopyParams& p, cudaStream_t stream) {
  constexpr int U = VEC == 32 ? (KV_COPY_UNROLL + 1) / 2 : KV_COPY_UNROLL;
  return launch(kv_copy_rows<VEC, U, IdxT>, p.shape.num_units, p, stream);
}

template <typename IdxT>
kv_status launch_copy(int vec, const CopyParams& p, cudaStream_t stream) {
  switch (vec) {
#if KV_MAX_VEC >= 32
    case 32: return launch_copy_vec<32, IdxT>(p, stream);
#endif
    case 16: return launch_copy_vec<16, IdxT>(p, stream);
    case 8: return launch_copy_vec<8, IdxT>(p, stream);
    case 4: return launch_copy_vec<4, IdxT>(p, stream);
    case 2: return launch_copy_vec<2, IdxT>(p, stream);
    default: return launch_copy_vec<1, IdxT>(p, stream);
  }
}

// Large FP8 writes pair the K and the V part of a token in one warp (measured:
// fp8 7.68 -> 7.53 us per call); small launches keep one side per warp.  The
// plain copies measured no gain from pairing (prefill 38.7 -> 39.1 us) and do
// not pair.
template <int OUT, typename IdxT, int FMT>
kv_status launch_fp8_fmt(bool bf16, const Fp8Params& p, cudaStream_t stream) {
  constexpr int U = OUT == 32 ? 1 : OUT == 16 ? KV_FP8_UNROLL : 4;
  if (KV_STORE_PAIR && p.shape.num_units >= KV_LARGE_LAUNCH_WARPS) {
    Fp8Params q = p;   // one warp per (token, segment, part): K and V together
    q.shape.units_per_token = q.shape.units_per_side;
    q.shape.num_units /= 2;
    if (q.dyn.work != nullptr) {
      if (bf16) return launch(kv_fp8_rows<OUT, U, 2, IdxT, true, FMT, true>, q.shape.num_units, q, stream);
      return launch(kv_fp8_rows<OUT, U, 2, IdxT, false, FMT, true>, q.shape.num_units, q, stream);
    }
    if (bf16) return launch(kv_fp8_rows<OUT, U, 2, IdxT, true, FMT, false>, q.shape.num_units, q, stream);
    return launch(kv_fp8_rows<OUT, U, 2, IdxT, false, FMT, false>, q.shape.num_units, q, stream);
  }
  if (p.dyn.work != nullptr) {
    if (bf16) return launch(kv_fp8_rows<OUT, U, 1, IdxT, true, FMT, true>, p.shape.num_units, p, stream);
    return launch(kv_fp8_rows<OUT, U, 1, IdxT, false, FMT, true>, p.shape.num_units, p, stream);
  }
  if (bf16) return launch(kv_fp8_rows<OUT, U, 1, IdxT, true, FMT, false>, p.shape.num_units, p, stream);
  return launch(kv_fp8_rows<OUT, U, 1, IdxT, false, FMT, false>, p.shape.num_units, p, stream);
}

template <int OUT, typename IdxT>
kv_status launch_fp8_out(int fmt, bool bf16, const Fp8Params& p, cudaStream_t stream) {
  if (fmt == kFmtE5M2) return launch_fp8_fmt<OUT, IdxT, kFmtE5M2>(bf16, p, stream);
  return launch_fp8_fmt<OUT, IdxT, kFmtE4M3>(bf16, p, stream);
}

template <typename IdxT>
kv_status launch_fp8(int out, int fmt, bool bf16, const Fp8Params& p, cudaStream_t stream) {
  switch (out) {
#if KV_MAX_VEC >= 32
    case 32: return launch_fp8_out<32, IdxT>(fmt, bf16, p, stream);
#endif
    case 16: return launch_fp8_out<16, IdxT>(fmt, bf16, p, stream);
    case 8: return launch_fp8_out<8, IdxT>(fmt, bf16, p, stream);
    case 4: return launch_fp8_out<4, IdxT>(fmt, bf16, p, stream);
    default: return launch_fp8_out<2, IdxT>(fmt, bf16, p, stream);
  }
}

template <typename IdxT, int FMT>
kv_status launch_fp8_elements_fmt(bool bf16, const GenericFp8Params& g, cudaStream_t stream) {
  if (bf16) return launch(kv_fp8_elements<IdxT, true, FMT>, g.num_units, g, stream);
  return launch(kv_fp8_elements<IdxT, false, FMT>, g.num_units, g, stream);
}

template <typename IdxT>
kv_status launch_fp8_elements(int fmt, bool bf16, const GenericFp8Params& g, cudaStream_t stream) {
  if (fmt == kFmtE5M2) return launch_fp8_elements_fmt<IdxT, kFmtE5M2>(bf16, g, stream);
  return launch_fp8_elements_fmt<IdxT, kFmtE4M3>(bf16, g, stream);
}

}  // namespace kvimpl

using namespace kvimpl;

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

namespace {

// kv_store and kv_store_paged: a plain copy into a flat (page_size 1) or paged cache.
kv_status store_copy(const void* k, const void* v, void* k_cache, void* v_cache,
                     const void* indices, kv_index_dtype index_dtype, int64_t index_stride,
                     int64_t num_tokens, int32_t num_heads, int32_t head_dim, int32_t elem_bytes,
                     const kv_strides* s, int64_t page_size, int64_t kc_page_stride,
                     int64_t vc_page_stride, int64_t size_limit, int32_t num_split,
                     kv_error_record* d_err, kv_stream_t stream_) {
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!common_args_ok(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_heads,
                      head_dim, s, size_limit, d_err))
    return KV_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return KV_ERR_INVALID_ARG;
  if (num_split != 0 && num_split != 1 && num_split != 2 && num_split != 4) return KV_ERR_INVALID_ARG;
  const int64_t row_bytes = static_cast<int64_t>(num_heads) * head_dim * elem_bytes;
  if (num_split > 1 && row_bytes % (static_cast<int64_t>(num_split) * 128) != 0)
    return KV_ERR_INVALID_ARG;
  if (page_size < 1) return KV_ERR_INVALID_ARG;
  // A page stride of page_size slots is the flat layout: slot * slot_stride.
  const bool flat = kc_page_stride == page_size * s->kc_slot && vc_page_stride == page_size * s->vc_slot;
  const int64_t psize = flat ? 1 : page_size;
  const int64_t kpage = flat ? s->kc_slot : kc_page_stride;
  const int64_t vpage = flat ? s->vc_slot : vc_page_stride;
  if (num_tokens > (int64_t{1} << 40)) return KV_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool i64 = index_dtype == KV_INDEX_I64;
  bool on_device = true;
  {
    const void* in[3] = {k, v, indices};
    const kv_status cs = classify_inputs(in, 3, &on_device);
    if (cs != KV_OK) return cs;
  }

  if (s->k_dim != elem_bytes || s->v_dim != elem_bytes || s->kc_dim != elem_bytes ||
      s->vc_dim != elem_bytes) {
    GenericCopyParams g = {};
    g.src[0] = static_cast<const uint8_t*>(k);
    g.src[1] = static_cast<const uint8_t*>(v);
    g.dst[0] = static_cast<uint8_t*>(k_cache);
    g.dst[1] = static_cast<uint8_t*>(v_cache);
    g.src_token[0] = s->k_token; g.src_head[0] = s->k_head; g.src_dim[0] = s->k_dim;
    g.src_token[1] = s->v_token; g.src_head[1] = s->v_head; g.src_dim[1] = s->v_dim;
    g.dst_slot[0] = s->kc_slot; g.dst_head[0] = s->kc_head; g.dst_dim[0] = s->kc_dim;
    g.dst_slot[1] = s->vc_slot; g.dst_head[1] = s->vc_head; g.dst_dim[1] = s->vc_dim;
    g.dst_page[0] = kpage;
    g.dst_page[1] = vpage;
    g.page_size = psize;
    g.indices = indices;
    g.index_stride = index_stride;
    g.size_limit = size_limit;
    g.num_units = static_cast<uint64_t>(num_tokens) * 2u * static_cast<uint64_t>(num_heads);
    g.num_heads = num_heads;
    g.head_dim = head_dim;
    g.elem_bytes = elem_bytes;
    g.err = d_err;
    return i64 ? launch(kv_copy_elements<int64_t>, g.num_units, g, stream)
               : launch(kv_copy_elements<int32_t>, g.num_units, g, stream);
  }

  const int64_t head_bytes = static_cast<int64_t>(head_dim) * elem_bytes;
  const Segments sg = segments(num_heads, head_dim, head_bytes, head_bytes, s);
  const int64_t seg_bytes = sg.elems * elem_bytes;
  uint64_t bits = u64(k) | u64(v) | u64(k_cache) | u64(v_cache) | u64(s->k_token) |
                  u64(s->v_token) | u64(s->kc_slot) | u64(s->vc_slot) | u64(seg_bytes);
  if (sg.count > 1) bits |= u64(s->k_head) | u64(s->v_head) | u64(s->kc_head) | u64(s->vc_head);
  if (!flat) bits |= u64(kc_page_stride) | u64(vc_page_stride);

  int sms = 0;
  kv_status st = current_sm_count(&sms);
  if (st != KV_OK) return st;
  uint32_t parts = 1;
  const uint64_t rows = static_cast<uint64_t>(num_tokens) * 2u * sg.count;
  if (num_split == 0) {
    const int vec0 = pow2_align(bits);
    parts = auto_parts(rows, seg_bytes / vec0, sms);
  } else if (num_split > 1 && seg_bytes % (num_split * 16) == 0) {
    parts = static_cast<uint32_t>(num_split);
  }
  const int64_t part_bytes = seg_bytes / parts;
  const int vec = pow2_align(bits | u64(part_bytes));

  CopyParams p = {};
  p.side[0] = CopySide{static_cast<const uint8_t*>(k), static_cast<uint8_t*>(k_cache), s->k_token,
                       s->k_head, s->kc_slot, s->kc_head, kpage};
  p.side[1] = CopySide{static_cast<const uint8_t*>(v), static_cast<uint8_t*>(v_cache), s->v_token,
                       s->v_head, s->vc_slot, s->vc_head, vpage};
  p.indices = indices;
  p.index_stride = index_stride;
  p.size_limit = size_limit;
  p.page_size = psize;
  p.shape.parts = parts;
  p.shape.units_per_side = sg.count * parts;
  p.shape.units_per_token = 2u * p.shape.units_per_side;
  p.shape.num_units = static_cast<uint64_t>(num_tokens) * p.shape.units_per_token;
  p.shape.part_chunks = static_cast<uint32_t>(part_bytes / vec);
  p.err = d_err;
  p.prefetch = vec >= 16 && on_device ? 1 : 0;
  p.vec = vec;
  return i64 ? launch_copy<int64_t>(vec, p, stream) : launch_copy<int32_t>(vec, p, stream);
}

}  // namespace

extern "C" kv_status kv_store(const void* k, const void* v, void* k_cache, void* v_cache,
                              const void* indices, kv_index_dtype index_dtype, int64_t index_stride,
                              int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                              int32_t elem_bytes, const kv_strides* s, int64_t size_limit,
                              int32_t num_split, kv_error_record* d_err, kv_stream_t stream) {
  const int64_t kpage = s != nullptr ? s->kc_slot : 0;
  const int64_t vpage = s != nullptr ? s->vc_slot : 0;
  return store_copy(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                    num_heads, head_dim, elem_bytes, s, 1, kpage, vpage, size_limit, num_split,
                    d_err, stream);
}

extern "C" kv_status kv_store_paged(const void* k, const void* v, void* k_cache, void* v_cache,
                                    const void* indices, kv_index_dtype index_dtype,
                                    int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                    int32_t head_dim, int32_t elem_bytes, const kv_strides* s,
                                    int64_t page_size, int64_t kc_page_stride,
                                    int64_t vc_page_stride, int64_t size_limit, int32_t num_split,
                                    kv_error_record* d_err, kv_stream_t stream) {
  return store_copy(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                    num_heads, head_dim, elem_bytes, s, page_size, kc_page_stride, vc_page_stride,
                    size_limit, num_split, d_err, stream);
}

// kv_store_fp8, and the static scale modes of kv_store_fp8_ex: one inverse
// scale per tensor (or none), or with scale_page > 0 one inverse scale per
// cache page (index slot / scale_page); output format fmt (kFmtE4M3 /
// kFmtE5M2).
kv_status kvimpl::store_fp8_static(const void* k, const void* v, void* k_cache, void* v_cache,
                                   const void* indices, kv_index_dtype index_dtype,
                                   int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                   int32_t head_dim, kv_src_dtype src_dtype, const kv_strides* s,
                                   int64_t page_size, int64_t kc_page_stride,
                                   int64_t vc_page_stride, int64_t size_limit,
                                   const float* inv_k_scale, const float* inv_v_scale,
                                   int32_t use_scale, int64_t scale_page, int fmt,
                                   kv_error_record* d_err, kv_stream_t stream_,
                                   const DynTensor* dyn) {
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!common_args_ok(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_heads,
                      head_dim, s, size_limit, d_err))
    return KV_ERR_INVALID_ARG;
  if (src_dtype != KV_SRC_F16 && src_dtype != KV_SRC_BF16) return KV_ERR_INVALID_ARG;
  if (page_size < 1) return KV_ERR_INVALID_ARG;
  if (dyn == nullptr && use_scale && (!inv_k_scale || !inv_v_scale)) return KV_ERR_INVALID_ARG;
  if (use_scale && ((u64(inv_k_scale) | u64(inv_v_scale)) & 3u) != 0) return KV_ERR_INVALID_ARG;
  if (scale_page < 0 || (scale_page != 0 && !use_scale)) return KV_ERR_INVALID_ARG;
  const uint64_t src_bits = u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token) | u64(s->k_head) |
                            u64(s->v_head) | u64(s->k_dim) | u64(s->v_dim);
  if ((src_bits & 1u) != 0) return KV_ERR_INVALID_ARG;
  if (num_tokens > (int64_t{1} << 40)) return KV_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool i64 = index_dtype == KV_INDEX_I64;
  const bool bf16 = src_dtype == KV_SRC_BF16;
  bool on_device = true;
  {
    const void* in[3] = {k, v, indices};
    const kv_status cs = classify_inputs(in, 3, &on_device);
    if (cs != KV_OK) return cs;
  }
  const float* inv_k = use_scale ? inv_k_scale : nullptr;
  const float* inv_v = use_scale ? inv_v_scale : nullptr;
  // A page stride equal to page_size slots is the flat 3-D layout: s * slot_stride.
  const bool flat = kc_page_stride == page_size * s->kc_slot && vc_page_stride == page_size * s->vc_slot;

  const bool contiguous = s->k_dim == 2 && s->v_dim == 2 && s->kc_dim == 1 && s->vc_dim == 1;
  Segments sg{0u, 0};
  int out = 1;
  if (contiguous) {
    sg = segments(num_heads, head_dim, 2 * static_cast<int64_t>(head_dim), head_dim, s);
    uint64_t dst_bits = u64(k_cache) | u64(v_cache) | u64(s->kc_slot) | u64(s->vc_slot) |
                        u64(sg.elems);
    uint64_t sbits = u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token);
    if (sg.count > 1) {
      dst_bits |= u64(s->kc_head) | u64(s->vc_head);
      sbits |= u64(s->k_head) | u64(s->v_head);
    }
    if (!flat) dst_bits |= u64(kc_page_stride) | u64(vc_page_stride);
    out = pow2_align(dst_bits);
    if (out > KV_FP8_MAX_OUT) out = KV_FP8_MAX_OUT;
    // an OUT-byte chunk reads 2*OUT input bytes with loads of at most KV_MAX_VEC bytes
    while (out > 1 &&
           (sbits & static_cast<uint64_t>((2 * out > KV_MAX_VEC ? KV_MAX_VEC : 2 * out) - 1)) != 0)
      out >>= 1;
  }

  if (out < 2) {
    GenericFp8Params g = {};
    g.src[0] = static_cast<const uint8_t*>(k);
    g.src[1] = static_cast<const uint8_t*>(v);
    g.dst[0] = static_cast<uint8_t*>(k_cache);
    g.dst[1] = static_cast<uint8_t*>(v_cache);
    g.src_token[0] = s->k_token; g.src_head[0] = s->k_head; g.src_dim[0] = s->k_dim;
    g.src_token[1] = s->v_token; g.src_head[1] = s->v_head; g.src_dim[1] = s->v_dim;
    g.dst_slot[0] = s->kc_slot; g.dst_head[0] = s->kc_head; g.dst_dim[0] = s->kc_dim;
    g.dst_slot[1] = s->vc_slot; g.dst_head[1] = s->vc_head; g.dst_dim[1] = s->vc_dim;
    g.dst_page[0] = flat ? s->kc_slot : kc_page_stride;
    g.dst_page[1] = flat ? s->vc_slot : vc_page_stride;
    g.page_size = flat ? 1 : page_size;
    g.inv[0] = inv_k;
    g.inv[1] = inv_v;
    g.scale_page = scale_page;
    g.indices = indices;
    g.index_stride = index_stride;
    g.size_limit = size_limit;
    g.num_units = static_cast<uint64_t>(num_tokens) * 2u * static_cast<uint64_t>(num_heads);
    g.num_heads = num_heads;
    g.head_dim = head_dim;
    g.err = d_err;
    if (dyn != nullptr) g.dyn = *dyn;
    return i64 ? launch_fp8_elements<int64_t>(fmt, bf16, g, stream)
               : launch_fp8_elements<int32_t>(fmt, bf16, g, stream);
  }

  int sms = 0;
  kv_status st = current_sm_count(&sms);
  if (st != KV_OK) return st;
  const uint64_t rows = static_cast<uint64_t>(num_tokens) * 2u * sg.count;
  uint32_t parts = auto_parts(rows, sg.elems / out, sms);
  const int64_t part_elems = sg.elems / parts;

  Fp8Params p = {};
  p.side[0] = Fp8Side{static_cast<const uint8_t*>(k), static_cast<uint8_t*>(k_cache), s->k_token,
                      s->k_head, s->kc_slot, s->kc_head, flat ? s->kc_slot : kc_page_stride, inv_k};
  p.side[1] = Fp8Side{static_cast<const uint8_t*>(v), static_cast<uint8_t*>(v_cache), s->v_token,
                      s->v_head, s->vc_slot, s->vc_head, flat ? s->vc_slot : vc_page_stride, inv_v};
  p.indices = indices;
  p.index_stride = index_stride;
  p.size_limit = size_limit;
  p.page_size = flat ? 1 : page_size;
  p.scale_page = scale_page;
  p.scale_page_shift = -1;
  if (scale_page > 0 && (scale_page & (scale_page - 1)) == 0) {
    p.scale_page_shift = 0;
    while ((int64_t{1} << p.scale_page_shift) < scale_page) ++p.scale_page_shift;
  }
  p.shape.parts = parts;
  p.shape.units_per_side = sg.count * parts;
  p.shape.units_per_token = 2u * p.shape.units_per_side;
  p.shape.num_units = static_cast<uint64_t>(num_tokens) * p.shape.units_per_token;
  p.shape.part_chunks = static_cast<uint32_t>(part_elems / out);
  p.err = d_err;
  p.prefetch = out >= 8 && on_device ? 1 : 0;  // 2*OUT input bytes per chunk, 16-byte aligned
  p.vec = out;
  if (dyn != nullptr) p.dyn = *dyn;
  return i64 ? launch_fp8<int64_t>(out, fmt, bf16, p, stream)
             : launch_fp8<int32_t>(out, fmt, bf16, p, stream);
}

extern "C" kv_status kv_store_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                                  const void* indices, kv_index_dtype index_dtype,
                                  int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                  int32_t head_dim, kv_src_dtype src_dtype, const kv_strides* s,
                                  int64_t page_size, int64_t kc_page_stride, int64_t vc_page_stride,
                                  int64_t size_limit, const float* inv_k_scale,
                                  const float* inv_v_scale, int32_t use_scale,
                                  kv_error_record* d_err, kv_stream_t stream) {
  return store_fp8_static(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                          num_heads, head_dim, src_dtype, s, page_size, kc_page_stride,
                          vc_page_stride, size_limit, inv_k_scale, inv_v_scale, use_scale, 0,
                          kFmtE4M3, d_err, stream);
}

extern "C" kv_status kv_store_fp8_dynamic_tensor(
    const void* k, const void* v, void* k_cache, void* v_cache, const void* indices,
    kv_index_dtype index_dtype, int64_t index_stride, int64_t num_tokens, int32_t num_heads,
    int32_t head_dim, kv_src_dtype src_dtype, const kv_strides* s, int64_t page_size,
    int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit, kv_fp8_format format,
    float* k_scale, float* v_scale, uint64_t* work, kv_error_record* d_err, kv_stream_t stream_) {
  // Every check the two launches make comes first: once the reduction has
  // run, the write must follow, or the workspace is left mid-call.
  if (format != KV_FP8_E4M3FN && format != KV_FP8_E5M2) return KV_ERR_INVALID_ARG;
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (!k_scale || !v_scale || !work || ((u64(k_scale) | u64(v_scale)) & 3u) != 0 ||
      (u64(work) & 7u) != 0)
    return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!common_args_ok(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_heads,
                      head_dim, s, size_limit, d_err))
    return KV_ERR_INVALID_ARG;
  if (src_dtype != KV_SRC_F16 && src_dtype != KV_SRC_BF16) return KV_ERR_INVALID_ARG;
  if (page_size < 1) return KV_ERR_INVALID_ARG;
  if (((u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token) | u64(s->k_head) | u64(s->v_head)) &
       1u) != 0)
    return KV_ERR_INVALID_ARG;
  if (s->k_dim != 2 || s->v_dim != 2) return KV_ERR_UNSUPPORTED;
  if (num_tokens > (int64_t{1} << 40)) return KV_ERR_UNSUPPORTED;
  // the workspace (64-bit atomics) and the scale outputs live in device memory
  const void* dev_only[3] = {work, k_scale, v_scale};
  for (const void* q : dev_only) {
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, q);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return cuda_fail(e);
    }
    if (a.type != cudaMemoryTypeDevice) return KV_ERR_INVALID_ARG;
  }
  bool on_device = true;
  {
    const void* in[3] = {k, v, indices};
    const kv_status cs = classify_inputs(in, 3, &on_device);
    if (cs != KV_OK) return cs;
  }
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  kv_status st = absmax_reduce(k, v, src_dtype, num_tokens, num_heads, head_dim, s, nullptr, work,
                               on_device, stream);
  if (st != KV_OK) return st;
  const DynTensor dyn{work, {k_scale, v_scale}, format == KV_FP8_E5M2 ? 57344.0f : 448.0f};
  return store_fp8_static(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                          num_heads, head_dim, src_dtype, s, page_size, kc_page_stride,
                          vc_page_stride, size_limit, nullptr, nullptr, 1, 0,
                          format == KV_FP8_E5M2 ? kFmtE5M2 : kFmtE4M3, d_err, stream_, &dyn);
}

extern "C" kv_status kv_error_poll(kv_error_record* d_err, kv_stream_t stream_, int64_t* oob_count,
                                   int64_t* first_bad_token) {
  if (!d_err || (u64(d_err) & 7u) != 0) return KV_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  kv_error_record h = {0, 0};
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpyAsync(&h, d_err, sizeof h, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemsetAsync(d_err, 0, sizeof h, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (oob_count) *oob_count = static_cast<int64_t>(h.oob_count);
  if (first_bad_token)
    *first_bad_token = h.oob_count ? static_cast<int64_t>(~h.first_bad_key) : int64_t{-1};
  return h.oob_count ? KV_ERR_INDEX_OOB : KV_OK;
}

namespace kvimpl {
namespace {

struct SnapshotParams {
  const kv_error_record* src;
  kv_error_record* dst;
};

// Copies the record after the preceding grid has finished (programmatic
// launch wait), so a captured step can hand its status to the host without a
// copy-engine round trip.
__global__ void __launch_bounds__(kThreads) kv_error_snapshot_kernel(const __grid_constant__ SnapshotParams p) {
  grid_handover<true>();  // small bookkeeping kernel: let the next kernel in early
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const unsigned long long n = *reinterpret_cast<const volatile unsigned long long*>(&p.src->oob_count);
    const unsigned long long f = *reinterpret_cast<const volatile unsigned long long*>(&p.src->first_bad_key);
    p.dst->oob_count = n;
    p.dst->first_bad_key = f;
  }
}

}  // namespace
}  // namespace kvimpl

extern "C" kv_status kv_error_snapshot(const kv_error_record* d_err, kv_error_record* dst,
                                       kv_stream_t stream_) {
  if (!d_err || !dst || ((u64(d_err) | u64(dst)) & 7u) != 0) return KV_ERR_INVALID_ARG;
  bool on_device = true;
  const void* ptrs[2] = {d_err, dst};
  const kv_status cs = classify_inputs(ptrs, 2, &on_device);
  if (cs != KV_OK) return cs;
  return launch(kv_error_snapshot_kernel, 1, SnapshotParams{d_err, dst},
                reinterpret_cast<cudaStream_t>(stream_));
}

namespace kvimpl {
namespace {

struct FloorParams {
  int unused;
};

// No memory access: the grid-dependency hand-over of the row kernels and
// nothing else.
__global__ void __launch_bounds__(kThreads) kv_launch_floor_kernel(const __grid_constant__ FloorParams) {
  grid_handover();
}

}  // namespace
}  // namespace kvimpl

extern "C" kv_status kv_launch_floor(int64_t num_warps, kv_stream_t stream_) {
  if (num_warps < 1 || num_warps > (int64_t{1} << 40)) return KV_ERR_INVALID_ARG;
  return launch(kv_launch_floor_kernel, static_cast<uint64_t>(num_warps), FloorParams{0},
                reinterpret_cast<cudaStream_t>(stream_));
}

extern "C" kv_status kv_error_reset(kv_error_record* d_err, kv_stream_t stream_) {
  if (!d_err || (u64(d_err) & 7u) != 0) return KV_ERR_INVALID_ARG;
  const cudaError_t e =
      cudaMemsetAsync(d_err, 0, sizeof(kv_error_record), reinterpret_cast<cudaStream_t>(stream_));
  if (e != cudaSuccess) return cuda_fail(e);
  return KV_OK;
}

extern "C" const char* kv_status_str(kv_status status) {
  switch (status) {
    case KV_OK: return "KV_OK";
    case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
    case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
    case KV_ERR_CUDA: return "KV_ERR_CUDA";
    case KV_ERR_INDEX_OOB: return "KV_ERR_INDEX_OOB";
  }
  return "KV_STATUS_UNKNOWN";
}

extern "C" int kv_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" int kv_abi_version(void) { return KV_ABI_VERSION; }

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory: kv_store with
// its error record in a static device array of this library.
// ---------------------------------------------------------------------------

namespace kvimpl {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KV_NOALLOC_SCRATCH_BYTES];
static_assert(sizeof(kv_error_record) <= KV_NOALLOC_SCRATCH_BYTES, "record must fit the array");

// Unique id of the calling thread's current CUDA context, or 0 when there is
// none yet (or the driver cannot tell).  The driver functions are fetched
// through the runtime, so the library does not link the driver library.
unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
    (void)cudaGetLastError();
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch for each device, looked up with that
// device current and kept together with the id of the context it belongs to.
// In host code the array's name is only a host-side stand-in.  A context
// that is not the one of the cached address (after cudaDeviceReset the
// runtime makes a new one, and the module, with the array, may then load
// elsewhere) or an unknown context leads to a fresh lookup.
struct NoallocAddr {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_noalloc_mutex;
NoallocAddr g_noalloc_addr[kMaxDevices];

kv_status noalloc_record(kv_error_record** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return KV_ERR_UNSUPPORTED;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocAddr& slot = g_noalloc_addr[dev];
  if (ctx == 0 || slot.addr == nullptr || slot.ctx_id != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    slot.addr = p;
    slot.ctx_id = current_context_id();  // the lookup has made the context current
  }
  *out = static_cast<kv_error_record*>(slot.addr);
  return KV_OK;
}

}  // namespace kvimpl

extern "C" kv_status kv_store_noalloc(const void* k, const void* v, void* k_cache, void* v_cache,
                                      const void* indices, kv_index_dtype index_dtype,
                                      int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                      int32_t head_dim, int32_t elem_bytes, const kv_strides* s,
                                      int64_t size_limit, int32_t num_split, int64_t* oob_count,
                                      int64_t* first_bad_token, kv_stream_t stream_) {
  if (oob_count) *oob_count = 0;
  if (first_bad_token) *first_bad_token = -1;
  if (sizeof(kv_error_record) > KV_NOALLOC_SCRATCH_BYTES) return KV_ERR_UNSUPPORTED;
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  kv_error_record* rec = nullptr;
  kv_status st = noalloc_record(&rec);
  if (st != KV_OK) return st;
  // The array keeps the previous call's counts: clear them first.
  cudaError_t e = cudaMemsetAsync(rec, 0, sizeof(kv_error_record), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  st = kv_store(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens, num_heads,
                head_dim, elem_bytes, s, size_limit, num_split, rec, stream_);
  if (st != KV_OK) return st;
  kv_error_record h = {0, 0};
  e = cudaMemcpyAsync(&h, rec, sizeof h, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (oob_count) *oob_count = static_cast<int64_t>(h.oob_count);
  if (first_bad_token && h.oob_count) *first_bad_token = static_cast<int64_t>(~h.first_bad_key);
  return h.oob_count ? KV_ERR_INDEX_OOB : KV_OK;
}
