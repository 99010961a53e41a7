// The inverse of the KV-cache write: gather cache rows back into token-major
// rows (kv_gather), optionally dequantising FP8 e4m3fn rows to bf16/fp16
// (kv_gather_fp8).  Row t of the outputs takes the cache row of slot
// indices[t].  This is the single-GPU counterpart of the materialise step of
// vLLM dcp_direct_kv_gather.cu (`materialize_kv_gather_kernel`, a vectorised
// copy of received KV into the caller's contiguous workspace); the
// cross-GPU multicast part of that page needs more than one GPU and is not
// here.
//
// Same decomposition as the write kernels: one warp per (token, K|V, segment,
// part) unit, lane l moving chunks l, l+32, ...  Here the source address
// depends on the slot, so the row loads follow the slot load.  Three things
// shorten that chain: before the programmatic-launch wait a warp reads its
// slot speculatively and prefetches the guessed rows into L2; large launches
// pair the K and the V part of a slot in one warp (one slot load for both);
// and in launches of more than one resident wave each warp also prefetches
// the rows of the unit one wave ahead.
#include "kv_host.h"

namespace kvimpl {
namespace {

struct GatherSide {
  const uint8_t* cache;  // element (slot 0, 0, 0) of the cache
  uint8_t* out;          // element (0, 0, 0) of the token-major output
  int64_t cache_slot, cache_seg, cache_page;
  int64_t out_token, out_seg;
  const float* scale;    // fp8, per-tensor mode: device scalar; per-page mode: one per page
  const float* scales;   // fp8, per-token / per-head modes: per-slot scale cache
};

struct GatherParams {
  GatherSide side[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size;
  UnitShape shape;
  kv_error_record* err;
  int vec;          // cache bytes per chunk
  int prefetch;     // cache rows are 16-byte aligned: speculative L2 prefetch allowed
  int scale_mode;   // fp8: kv_scale_mode (per-head mode: one head per unit segment)
  int64_t scales_stride;  // per-slot modes: floats per slot; per-page mode: the page size
  uint64_t ahead;   // > 0: also prefetch the cache rows of unit u + ahead (set by launch_rows)
};

// Dequantisation multiplier of a unit (fp8 gathers).
__device__ __forceinline__ float unit_scale(const GatherParams& p, const GatherSide& sd,
                                            int64_t slot, uint32_t seg) {
  switch (p.scale_mode) {
    case KV_SCALE_TENSOR: return __ldg(sd.scale);
    case KV_SCALE_TOKEN: return __ldg(sd.scales + slot * p.scales_stride);
    case KV_SCALE_TOKEN_HEAD: return __ldg(sd.scales + slot * p.scales_stride + seg);
    case KV_SCALE_PAGE: return __ldg(sd.scale + slot / p.scales_stride);
    default: return 1.0f;
  }
}


__device__ __forceinline__ int64_t gather_slot_offset(const GatherParams& p, const GatherSide& sd,
                                                      int64_t slot) {
  if (p.page_size == 1) return slot * sd.cache_page;
  const int64_t page = slot / p.page_size;
  return page * sd.cache_page + (slot - page * p.page_size) * sd.cache_slot;
}

// L2 prefetch of unit w's cache row part (of both sides when NS == 2) at
// slot s, when s is in range.
template <int NS>
__device__ __forceinline__ void gather_prefetch_rows(const GatherParams& p, const Unit& w, int64_t s) {
  if (s < 0 || s >= p.size_limit) return;
  const int64_t part_bytes = static_cast<int64_t>(p.shape.part_chunks) * p.vec;
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const GatherSide& sd = p.side[NS == 2 ? i : w.kv];
    prefetch_l2_bulk(sd.cache + gather_slot_offset(p, sd, s) +
                         static_cast<int64_t>(w.seg) * sd.cache_seg +
                         static_cast<int64_t>(w.part) * part_bytes,
                     static_cast<uint32_t>(part_bytes));
  }
}

// Before the wait: guess the unit's slot and prefetch its rows.
template <int NS, typename IdxT>
__device__ __forceinline__ void gather_prefetch(const GatherParams& p, const Unit& w) {
  gather_prefetch_rows<NS>(p, w, speculative_slot<IdxT>(p.indices, p.index_stride, w.token));
}

// After the wait, before moving unit u: lane 0 reads the slot of unit
// u + ahead (the unit a warp will take one resident wave later) and, once
// the unit's own loads are issued, prefetches that unit's rows into L2.
// Only the paired form (NS == 2) does this: multi-wave launches are large,
// and large launches pair; the small one-side launches keep their code.
struct Lookahead {
  Unit w{};
  int64_t slot = -1;
};

template <int NS, typename IdxT>
__device__ __forceinline__ Lookahead lookahead_slot(const GatherParams& p, uint64_t u, uint32_t lane) {
  Lookahead a;
  if (KV_LOOKAHEAD && NS == 2 && p.ahead != 0 && lane == 0 && u + p.ahead < p.shape.num_units) {
    a.w = decode_unit(p.shape, u + p.ahead);
    a.slot = load_slot<IdxT>(p.indices, p.index_stride, a.w.token);
  }
  return a;
}

// One unit of a gather: the slot is read once; NS == 2 moves the K and the V
// part of the unit (one slot load for both), NS == 1 the side w.kv.
template <int VEC, int U, int NS, typename IdxT>
__device__ __forceinline__ void gather_unit(const GatherParams& p, const Unit& w, uint32_t lane) {
  const uint32_t nchunks = p.shape.part_chunks;
  const int64_t part_bytes = static_cast<int64_t>(nchunks) * VEC;
  const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, w.token);
  if (slot < 0 || slot >= p.size_limit) {
    if (w.rank == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(w.token));
    return;
  }
  const uint8_t* src[NS];
  uint8_t* dst[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const GatherSide& sd = p.side[NS == 2 ? i : w.kv];
    src[i] = sd.cache + gather_slot_offset(p, sd, slot) + static_cast<int64_t>(w.seg) * sd.cache_seg +
             static_cast<int64_t>(w.part) * part_bytes;
    dst[i] = sd.out + w.token * sd.out_token + static_cast<int64_t>(w.seg) * sd.out_seg +
             static_cast<int64_t>(w.part) * part_bytes;
  }
  Chunk<VEC> buf[NS][U];
  for (uint32_t c0 = 0; c0 < nchunks; c0 += 32u * U) {
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + lane + 32u * j;
        if (c < nchunks) ld_stream(buf[i][j], src[i] + static_cast<size_t>(c) * VEC);
      }
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + lane + 32u * j;
        if (c < nchunks) st_stream(dst[i] + static_cast<size_t>(c) * VEC, buf[i][j]);
      }
  }
}

template <int VEC, int U, int NS, typename IdxT>
__global__ void __launch_bounds__(kThreads) kv_gather_rows(const __grid_constant__ GatherParams p) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
  const bool active = u < p.shape.num_units;
  Unit w = decode_unit(p.shape, active ? u : 0);
  if (KV_PREFETCH && lane == 0 && active) {
    if (p.prefetch) gather_prefetch<NS, IdxT>(p, w);
    else prefetch_l2_line(static_cast<const IdxT*>(p.indices) + w.token * p.index_stride);
  }
  grid_handover();
  while (u < p.shape.num_units) {
    const Lookahead next = lookahead_slot<NS, IdxT>(p, u, lane);
    gather_unit<VEC, U, NS, IdxT>(p, w, lane);
    if (KV_LOOKAHEAD && NS == 2 && lane == 0) gather_prefetch_rows<NS>(p, next.w, next.slot);
    u += nwarps;
    if (u >= p.shape.num_units) break;
    w = decode_unit(p.shape, u);
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// ---------------------------------------------------------------------------
// FP8 dequantising gather
// ---------------------------------------------------------------------------

// Two FP8 codes (lo in bits 0-7) to two fp32 values, exactly.  Every e4m3fn
// value is an fp16 value (hardware conversion); an e5m2 code is the top byte
// of the fp16 with the same value; fp16 widens exactly to fp32.
template <int FMT>
__device__ __forceinline__ float2 fp8x2_to_f32x2(uint32_t codes16) {
  uint32_t h2;
  if constexpr (FMT == kFmtE5M2) {
    h2 = ((codes16 & 0xFFu) << 8) | ((codes16 & 0xFF00u) << 16);
  } else {
    const uint16_t c = static_cast<uint16_t>(codes16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  }
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))));
}

// Two fp32 values to two bf16 / fp16 (lo in bits 0-15), nearest even.
template <bool kBF16>
__device__ __forceinline__ uint32_t narrow2(float lo, float hi) {
  uint32_t r;
  if constexpr (kBF16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// Four codes (one 32-bit word) to four 2-byte outputs (two words).
template <bool kBF16, int FMT>
__device__ __forceinline__ void dequant4(uint32_t codes, float scale, uint32_t& o0, uint32_t& o1) {
  const float2 a = fp8x2_to_f32x2<FMT>(codes & 0xFFFFu);
  const float2 b = fp8x2_to_f32x2<FMT>(codes >> 16);
  const float2 ya = mul2_rn(a, scale);
  const float2 yb = mul2_rn(b, scale);
  o0 = narrow2<kBF16>(ya.x, ya.y);
  o1 = narrow2<kBF16>(yb.x, yb.y);
}

// IN cache bytes (codes) per lane chunk -> 2*IN output bytes; NS as in
// gather_unit.
template <int IN, int U, int NS, typename IdxT, bool kBF16, int FMT>
__device__ __forceinline__ void gather_fp8_unit(const GatherParams& p, const Unit& w,
                                                uint32_t lane) {
  const uint32_t nchunks = p.shape.part_chunks;
  const int64_t part_in = static_cast<int64_t>(nchunks) * IN;
  const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, w.token);
  if (slot < 0 || slot >= p.size_limit) {
    if (w.rank == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(w.token));
    return;
  }
  const uint8_t* src[NS];
  uint8_t* dst[NS];
  float scale[NS];
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const GatherSide& sd = p.side[NS == 2 ? i : w.kv];
    scale[i] = unit_scale(p, sd, slot, w.seg);
    src[i] = sd.cache + gather_slot_offset(p, sd, slot) + static_cast<int64_t>(w.seg) * sd.cache_seg +
             static_cast<int64_t>(w.part) * part_in;
    dst[i] = sd.out + w.token * sd.out_token + static_cast<int64_t>(w.seg) * sd.out_seg +
             static_cast<int64_t>(w.part) * part_in * 2;
  }
  constexpr int kWords = IN >= 4 ? IN / 4 : 1;
  Chunk<IN> buf[NS][U];
  for (uint32_t c0 = 0; c0 < nchunks; c0 += 32u * U) {
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + lane + 32u * j;
        if (c < nchunks) ld_stream(buf[i][j], src[i] + static_cast<size_t>(c) * IN);
      }
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const uint32_t c = c0 + lane + 32u * j;
        if (c >= nchunks) continue;
        uint8_t* o = dst[i] + static_cast<size_t>(c) * (2 * IN);
        if constexpr (IN >= 4) {
          Chunk<2 * IN> out;
#pragma unroll
          for (int q = 0; q < kWords; ++q)
            dequant4<kBF16, FMT>(buf[i][j].w[q], scale[i], out.w[2 * q], out.w[2 * q + 1]);
          st_stream(o, out);
        } else {
          static_assert(IN == 2, "IN");
          const float2 a = fp8x2_to_f32x2<FMT>(buf[i][j].h);
          Chunk<4> out;
          out.w[0] = narrow2<kBF16>(__fmul_rn(a.x, scale[i]), __fmul_rn(a.y, scale[i]));
          st_stream(o, out);
        }
      }
  }
}

template <int IN, int U, int NS, typename IdxT, bool kBF16, int FMT>
__global__ void __launch_bounds__(kThreads) kv_gather_fp8_rows(const __grid_constant__ GatherParams p) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
  const bool active = u < p.shape.num_units;
  Unit w = decode_unit(p.shape, active ? u : 0);
  if (KV_PREFETCH && lane == 0 && active) {
    if (p.prefetch) gather_prefetch<NS, IdxT>(p, w);
    else prefetch_l2_line(static_cast<const IdxT*>(p.indices) + w.token * p.index_stride);
  }
  grid_handover();
  while (u < p.shape.num_units) {
    const Lookahead next = lookahead_slot<NS, IdxT>(p, u, lane);
    gather_fp8_unit<IN, U, NS, IdxT, kBF16, FMT>(p, w, lane);
    if (KV_LOOKAHEAD && NS == 2 && lane == 0) gather_prefetch_rows<NS>(p, next.w, next.slot);
    u += nwarps;
    if (u >= p.shape.num_units) break;
    w = decode_unit(p.shape, u);
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// Element-wise gathers for non-contiguous dims or odd sizes: one warp per
// (token, K|V, head), lanes over the head's elements.
struct GatherElemParams {
  const uint8_t* cache[2];
  uint8_t* out[2];
  int64_t cache_slot[2], cache_head[2], cache_dim[2], cache_page[2];
  int64_t out_token[2], out_head[2], out_dim[2];
  const float* scale[2];
  const float* scales[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size, scales_stride;
  uint64_t num_units;
  int32_t num_heads, head_dim, elem_bytes;  // elem_bytes: copy only
  int scale_mode;                           // fp8 only
  kv_error_record* err;
};

template <typename IdxT, int kMode, int FMT>  // kMode: 0 copy, 1 fp8 -> bf16, 2 fp8 -> fp16
__global__ void __launch_bounds__(kThreads) kv_gather_elements(const __grid_constant__ GatherElemParams p) {
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
    int64_t row;
    if (p.page_size == 1) {
      row = slot * p.cache_page[kv];
    } else {
      const int64_t page = slot / p.page_size;
      row = page * p.cache_page[kv] + (slot - page * p.page_size) * p.cache_slot[kv];
    }
    const uint8_t* src = p.cache[kv] + row + h * p.cache_head[kv];
    uint8_t* dst = p.out[kv] + t * p.out_token[kv] + h * p.out_head[kv];
    float scale = 1.0f;
    if (kMode != 0) {
      if (p.scale_mode == KV_SCALE_TENSOR) scale = __ldg(p.scale[kv]);
      else if (p.scale_mode == KV_SCALE_TOKEN) scale = __ldg(p.scales[kv] + slot * p.scales_stride);
      else if (p.scale_mode == KV_SCALE_TOKEN_HEAD)
        scale = __ldg(p.scales[kv] + slot * p.scales_stride + h);
      else if (p.scale_mode == KV_SCALE_PAGE)
        scale = __ldg(p.scale[kv] + slot / p.scales_stride);
    }
    for (int64_t d = lane; d < p.head_dim; d += 32) {
      const uint8_t* s = src + d * p.cache_dim[kv];
      uint8_t* o = dst + d * p.out_dim[kv];
      if constexpr (kMode == 0) {
        for (int b = 0; b < p.elem_bytes; ++b) o[b] = __ldg(s + b);
      } else {
        const float2 x = fp8x2_to_f32x2<FMT>(__ldg(s));
        const uint32_t v = narrow2<kMode == 1>(__fmul_rn(x.x, scale), 0.0f);
        o[0] = static_cast<uint8_t>(v & 0xFFu);
        o[1] = static_cast<uint8_t>((v >> 8) & 0xFFu);
      }
    }
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// Sides moved per warp by the row gathers: large launches pair the K and the V
// part of a slot in one warp (one slot load, twice the bytes in flight per
// dependent load); small, latency-bound launches keep one side per warp so
// that more warps share the round trips.  Rewrites the shape for pairing.
inline int gather_sides(GatherParams& p) {
  const bool pair = KV_GATHER_PAIR == 2 ||
                    (KV_GATHER_PAIR == 1 && p.shape.num_units >= KV_LARGE_LAUNCH_WARPS);
  if (!pair) return 1;
  p.shape.units_per_token = p.shape.units_per_side;
  p.shape.num_units /= 2;
  return 2;
}

// Bytes a gather launch moves: every unit's part read from the cache and
// written out (an FP8 unit writes out_per_in bytes per code).
inline uint64_t gather_bytes(const GatherParams& p, uint64_t out_per_in) {
  return p.shape.num_units * p.shape.part_chunks * static_cast<uint64_t>(p.vec) * (1 + out_per_in);
}

template <int VEC, typename IdxT>
kv_status launch_gather_vec(GatherParams p, cudaStream_t stream) {
  constexpr int U = VEC == 32 ? (KV_COPY_UNROLL + 1) / 2 : KV_COPY_UNROLL;
  const uint64_t bytes = gather_bytes(p, 1);
  if (gather_sides(p) == 2)
    return launch_rows(kv_gather_rows<VEC, U, 2, IdxT>, p.shape.num_units, p, stream, bytes);
  return launch_rows(kv_gather_rows<VEC, U, 1, IdxT>, p.shape.num_units, p, stream, bytes);
}

template <typename IdxT>
kv_status launch_gather(int vec, const GatherParams& p, cudaStream_t stream) {
  switch (vec) {
#if KV_MAX_VEC >= 32
    case 32: return launch_gather_vec<32, IdxT>(p, stream);
#endif
    case 16: return launch_gather_vec<16, IdxT>(p, stream);
    case 8: return launch_gather_vec<8, IdxT>(p, stream);
    case 4: return launch_gather_vec<4, IdxT>(p, stream);
    case 2: return launch_gather_vec<2, IdxT>(p, stream);
    default: return launch_gather_vec<1, IdxT>(p, stream);
  }
}

template <int IN, typename IdxT, int FMT>
kv_status launch_gather_fp8_fmt(bool bf16, const GatherParams& p, cudaStream_t stream) {
  constexpr int U = IN == 16 ? 2 : 4;
  const uint64_t bytes = gather_bytes(p, 2);
  GatherParams q = p;
  if (gather_sides(q) == 2) {
    if (bf16)
      return launch_rows(kv_gather_fp8_rows<IN, U, 2, IdxT, true, FMT>, q.shape.num_units, q, stream, bytes);
    return launch_rows(kv_gather_fp8_rows<IN, U, 2, IdxT, false, FMT>, q.shape.num_units, q, stream, bytes);
  }
  if (bf16)
    return launch_rows(kv_gather_fp8_rows<IN, U, 1, IdxT, true, FMT>, p.shape.num_units, p, stream, bytes);
  return launch_rows(kv_gather_fp8_rows<IN, U, 1, IdxT, false, FMT>, p.shape.num_units, p, stream, bytes);
}

template <int IN, typename IdxT>
kv_status launch_gather_fp8_in(int fmt, bool bf16, const GatherParams& p, cudaStream_t stream) {
  if (fmt == kFmtE5M2) return launch_gather_fp8_fmt<IN, IdxT, kFmtE5M2>(bf16, p, stream);
  return launch_gather_fp8_fmt<IN, IdxT, kFmtE4M3>(bf16, p, stream);
}

template <typename IdxT>
kv_status launch_gather_fp8(int in, int fmt, bool bf16, const GatherParams& p, cudaStream_t stream) {
  switch (in) {
    case 16: return launch_gather_fp8_in<16, IdxT>(fmt, bf16, p, stream);
    case 8: return launch_gather_fp8_in<8, IdxT>(fmt, bf16, p, stream);
    case 4: return launch_gather_fp8_in<4, IdxT>(fmt, bf16, p, stream);
    default: return launch_gather_fp8_in<2, IdxT>(fmt, bf16, p, stream);
  }
}

template <typename IdxT, int FMT>
kv_status launch_gather_elements_fmt(int mode, const GatherElemParams& g, cudaStream_t stream) {
  if (mode == 0) return launch(kv_gather_elements<IdxT, 0, FMT>, g.num_units, g, stream);
  if (mode == 1) return launch(kv_gather_elements<IdxT, 1, FMT>, g.num_units, g, stream);
  return launch(kv_gather_elements<IdxT, 2, FMT>, g.num_units, g, stream);
}

template <typename IdxT>
kv_status launch_gather_elements(int mode, int fmt, const GatherElemParams& g, cudaStream_t stream) {
  if (fmt == kFmtE5M2) return launch_gather_elements_fmt<IdxT, kFmtE5M2>(mode, g, stream);
  return launch_gather_elements_fmt<IdxT, kFmtE4M3>(mode, g, stream);
}

GatherElemParams element_params(const void* k_cache, const void* v_cache, void* k_out, void* v_out,
                                const void* indices, int64_t index_stride, int64_t num_tokens,
                                int32_t num_heads, int32_t head_dim, const kv_strides* s,
                                int64_t size_limit, kv_error_record* d_err) {
  GatherElemParams g = {};
  g.cache[0] = static_cast<const uint8_t*>(k_cache);
  g.cache[1] = static_cast<const uint8_t*>(v_cache);
  g.out[0] = static_cast<uint8_t*>(k_out);
  g.out[1] = static_cast<uint8_t*>(v_out);
  g.cache_slot[0] = s->kc_slot; g.cache_head[0] = s->kc_head; g.cache_dim[0] = s->kc_dim;
  g.cache_slot[1] = s->vc_slot; g.cache_head[1] = s->vc_head; g.cache_dim[1] = s->vc_dim;
  g.cache_page[0] = s->kc_slot;
  g.cache_page[1] = s->vc_slot;
  g.out_token[0] = s->k_token; g.out_head[0] = s->k_head; g.out_dim[0] = s->k_dim;
  g.out_token[1] = s->v_token; g.out_head[1] = s->v_head; g.out_dim[1] = s->v_dim;
  g.indices = indices;
  g.index_stride = index_stride;
  g.size_limit = size_limit;
  g.page_size = 1;
  g.num_units = static_cast<uint64_t>(num_tokens) * 2u * static_cast<uint64_t>(num_heads);
  g.num_heads = num_heads;
  g.head_dim = head_dim;
  g.err = d_err;
  return g;
}

}  // namespace
}  // namespace kvimpl

using namespace kvimpl;

namespace {

// kv_gather and kv_gather_paged.
kv_status gather_copy(const void* k_cache, const void* v_cache, void* k_out, void* v_out,
                      const void* indices, kv_index_dtype index_dtype, int64_t index_stride,
                      int64_t num_tokens, int32_t num_heads, int32_t head_dim, int32_t elem_bytes,
                      const kv_strides* s, int64_t page_size, int64_t kc_page_stride,
                      int64_t vc_page_stride, int64_t size_limit, kv_error_record* d_err,
                      kv_stream_t stream_) {
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!common_args_ok(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                      num_heads, head_dim, s, size_limit, d_err))
    return KV_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return KV_ERR_INVALID_ARG;
  if (page_size < 1) return KV_ERR_INVALID_ARG;
  const bool flat = kc_page_stride == page_size * s->kc_slot && vc_page_stride == page_size * s->vc_slot;
  if (num_tokens > (int64_t{1} << 40)) return KV_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool i64 = index_dtype == KV_INDEX_I64;
  bool on_device = true;
  {
    const void* in[5] = {k_cache, v_cache, indices, k_out, v_out};
    const kv_status cs = classify_inputs(in, 5, &on_device);
    if (cs != KV_OK) return cs;
  }

  if (s->k_dim != elem_bytes || s->v_dim != elem_bytes || s->kc_dim != elem_bytes ||
      s->vc_dim != elem_bytes) {
    GatherElemParams g = element_params(k_cache, v_cache, k_out, v_out, indices, index_stride,
                                        num_tokens, num_heads, head_dim, s, size_limit, d_err);
    g.elem_bytes = elem_bytes;
    g.cache_page[0] = flat ? s->kc_slot : kc_page_stride;
    g.cache_page[1] = flat ? s->vc_slot : vc_page_stride;
    g.page_size = flat ? 1 : page_size;
    return i64 ? launch_gather_elements<int64_t>(0, kFmtE4M3, g, stream)
               : launch_gather_elements<int32_t>(0, kFmtE4M3, g, stream);
  }
  const int64_t head_bytes = static_cast<int64_t>(head_dim) * elem_bytes;
  const Segments sg = segments(num_heads, head_dim, head_bytes, head_bytes, s);
  const int64_t seg_bytes = sg.elems * elem_bytes;
  uint64_t bits = u64(k_cache) | u64(v_cache) | u64(k_out) | u64(v_out) | u64(s->k_token) |
                  u64(s->v_token) | u64(s->kc_slot) | u64(s->vc_slot) | u64(seg_bytes);
  if (sg.count > 1) bits |= u64(s->k_head) | u64(s->v_head) | u64(s->kc_head) | u64(s->vc_head);
  if (!flat) bits |= u64(kc_page_stride) | u64(vc_page_stride);
  int sms = 0;
  kv_status st = current_sm_count(&sms);
  if (st != KV_OK) return st;
  const int vec0 = pow2_align(bits);
  const uint64_t rows = static_cast<uint64_t>(num_tokens) * 2u * sg.count;
  const uint32_t parts = auto_parts(rows, seg_bytes / vec0, sms);
  const int64_t part_bytes = seg_bytes / parts;
  const int vec = pow2_align(bits | u64(part_bytes));

  GatherParams p = {};
  p.side[0] = GatherSide{static_cast<const uint8_t*>(k_cache), static_cast<uint8_t*>(k_out),
                         s->kc_slot, s->kc_head, flat ? s->kc_slot : kc_page_stride, s->k_token,
                         s->k_head, nullptr, nullptr};
  p.side[1] = GatherSide{static_cast<const uint8_t*>(v_cache), static_cast<uint8_t*>(v_out),
                         s->vc_slot, s->vc_head, flat ? s->vc_slot : vc_page_stride, s->v_token,
                         s->v_head, nullptr, nullptr};
  p.indices = indices;
  p.index_stride = index_stride;
  p.size_limit = size_limit;
  p.page_size = flat ? 1 : page_size;
  p.shape.parts = parts;
  p.shape.units_per_side = sg.count * parts;
  p.shape.units_per_token = 2u * p.shape.units_per_side;
  p.shape.num_units = static_cast<uint64_t>(num_tokens) * p.shape.units_per_token;
  p.shape.part_chunks = static_cast<uint32_t>(part_bytes / vec);
  p.err = d_err;
  p.vec = vec;
  p.prefetch = vec >= 16 && on_device ? 1 : 0;
  return i64 ? launch_gather<int64_t>(vec, p, stream) : launch_gather<int32_t>(vec, p, stream);
}

}  // namespace

extern "C" kv_status kv_gather(const void* k_cache, const void* v_cache, void* k_out, void* v_out,
                               const void* indices, kv_index_dtype index_dtype, int64_t index_stride,
                               int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                               int32_t elem_bytes, const kv_strides* s, int64_t size_limit,
                               kv_error_record* d_err, kv_stream_t stream) {
  const int64_t kpage = s != nullptr ? s->kc_slot : 0;
  const int64_t vpage = s != nullptr ? s->vc_slot : 0;
  return gather_copy(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                     num_tokens, num_heads, head_dim, elem_bytes, s, 1, kpage, vpage, size_limit,
                     d_err, stream);
}

extern "C" kv_status kv_gather_paged(const void* k_cache, const void* v_cache, void* k_out,
                                     void* v_out, const void* indices, kv_index_dtype index_dtype,
                                     int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                     int32_t head_dim, int32_t elem_bytes, const kv_strides* s,
                                     int64_t page_size, int64_t kc_page_stride,
                                     int64_t vc_page_stride, int64_t size_limit,
                                     kv_error_record* d_err, kv_stream_t stream) {
  return gather_copy(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                     num_tokens, num_heads, head_dim, elem_bytes, s, page_size, kc_page_stride,
                     vc_page_stride, size_limit, d_err, stream);
}

namespace {

// kv_gather_fp8 and kv_gather_fp8_ex.
kv_status gather_fp8(const void* k_cache, const void* v_cache, void* k_out, void* v_out,
                     const void* indices, kv_index_dtype index_dtype, int64_t index_stride,
                     int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                     kv_src_dtype out_dtype, const kv_strides* s, int64_t page_size,
                     int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit, int fmt,
                     int scale_mode, const float* k_scale, const float* v_scale,
                     const float* k_scales, const float* v_scales, int64_t scales_stride,
                     kv_error_record* d_err, kv_stream_t stream_) {
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!common_args_ok(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                      num_heads, head_dim, s, size_limit, d_err))
    return KV_ERR_INVALID_ARG;
  if (out_dtype != KV_SRC_F16 && out_dtype != KV_SRC_BF16) return KV_ERR_INVALID_ARG;
  if (page_size < 1) return KV_ERR_INVALID_ARG;
  if ((scale_mode == KV_SCALE_TENSOR || scale_mode == KV_SCALE_PAGE) &&
      (!k_scale || !v_scale || ((u64(k_scale) | u64(v_scale)) & 3u) != 0))
    return KV_ERR_INVALID_ARG;
  if (scale_mode == KV_SCALE_PAGE) scales_stride = page_size;  // the scale index is slot / page_size
  const bool per_slot = scale_mode == KV_SCALE_TOKEN || scale_mode == KV_SCALE_TOKEN_HEAD;
  if (per_slot && (!k_scales || !v_scales || ((u64(k_scales) | u64(v_scales)) & 3u) != 0 ||
                   scales_stride < (scale_mode == KV_SCALE_TOKEN_HEAD ? num_heads : 1)))
    return KV_ERR_INVALID_ARG;
  const uint64_t out_bits = u64(k_out) | u64(v_out) | u64(s->k_token) | u64(s->v_token) |
                            u64(s->k_head) | u64(s->v_head) | u64(s->k_dim) | u64(s->v_dim);
  if ((out_bits & 1u) != 0) return KV_ERR_INVALID_ARG;
  if (num_tokens > (int64_t{1} << 40)) return KV_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool i64 = index_dtype == KV_INDEX_I64;
  const bool bf16 = out_dtype == KV_SRC_BF16;
  bool on_device = true;
  {
    const void* in[5] = {k_cache, v_cache, indices, k_out, v_out};
    const kv_status cs = classify_inputs(in, 5, &on_device);
    if (cs != KV_OK) return cs;
  }
  const bool one_scale_ptr = scale_mode == KV_SCALE_TENSOR || scale_mode == KV_SCALE_PAGE;
  const float* sk = one_scale_ptr ? k_scale : nullptr;
  const float* sv = one_scale_ptr ? v_scale : nullptr;
  const bool flat = kc_page_stride == page_size * s->kc_slot && vc_page_stride == page_size * s->vc_slot;
  const bool contiguous = s->k_dim == 2 && s->v_dim == 2 && s->kc_dim == 1 && s->vc_dim == 1;

  Segments sg{0u, 0};
  int in = 1;
  if (contiguous) {
    sg = segments(num_heads, head_dim, 2 * static_cast<int64_t>(head_dim), head_dim, s);
    if (scale_mode == KV_SCALE_TOKEN_HEAD)  // one head per unit: its segment index is the head
      sg = Segments{static_cast<uint32_t>(num_heads), static_cast<int64_t>(head_dim)};
    uint64_t cache_bits = u64(k_cache) | u64(v_cache) | u64(s->kc_slot) | u64(s->vc_slot) |
                          u64(sg.elems);
    uint64_t obits = u64(k_out) | u64(v_out) | u64(s->k_token) | u64(s->v_token);
    if (sg.count > 1) {
      cache_bits |= u64(s->kc_head) | u64(s->vc_head);
      obits |= u64(s->k_head) | u64(s->v_head);
    }
    if (!flat) cache_bits |= u64(kc_page_stride) | u64(vc_page_stride);
    in = pow2_align(cache_bits);
    if (in > KV_MAX_VEC / 2) in = KV_MAX_VEC / 2;  // the 2*IN output bytes fit one vector
    // an IN-byte chunk writes 2*IN output bytes with stores of at most KV_MAX_VEC bytes
    while (in > 1 &&
           (obits & static_cast<uint64_t>((2 * in > KV_MAX_VEC ? KV_MAX_VEC : 2 * in) - 1)) != 0)
      in >>= 1;
  }

  if (in < 2) {
    GatherElemParams g = element_params(k_cache, v_cache, k_out, v_out, indices, index_stride,
                                        num_tokens, num_heads, head_dim, s, size_limit, d_err);
    g.cache_page[0] = flat ? s->kc_slot : kc_page_stride;
    g.cache_page[1] = flat ? s->vc_slot : vc_page_stride;
    g.page_size = flat ? 1 : page_size;
    g.scale[0] = sk;
    g.scale[1] = sv;
    g.scales[0] = k_scales;
    g.scales[1] = v_scales;
    g.scales_stride = scales_stride;
    g.scale_mode = scale_mode;
    return i64 ? launch_gather_elements<int64_t>(bf16 ? 1 : 2, fmt, g, stream)
               : launch_gather_elements<int32_t>(bf16 ? 1 : 2, fmt, g, stream);
  }

  int sms = 0;
  kv_status st = current_sm_count(&sms);
  if (st != KV_OK) return st;
  const uint64_t rows = static_cast<uint64_t>(num_tokens) * 2u * sg.count;
  const uint32_t parts = auto_parts(rows, sg.elems / in, sms);
  const int64_t part_elems = sg.elems / parts;

  GatherParams p = {};
  p.side[0] = GatherSide{static_cast<const uint8_t*>(k_cache), static_cast<uint8_t*>(k_out),
                         s->kc_slot, s->kc_head, flat ? s->kc_slot : kc_page_stride, s->k_token,
                         s->k_head, sk, k_scales};
  p.side[1] = GatherSide{static_cast<const uint8_t*>(v_cache), static_cast<uint8_t*>(v_out),
                         s->vc_slot, s->vc_head, flat ? s->vc_slot : vc_page_stride, s->v_token,
                         s->v_head, sv, v_scales};
  p.indices = indices;
  p.index_stride = index_stride;
  p.size_limit = size_limit;
  p.page_size = flat ? 1 : page_size;
  p.shape.parts = parts;
  p.shape.units_per_side = sg.count * parts;
  p.shape.units_per_token = 2u * p.shape.units_per_side;
  p.shape.num_units = static_cast<uint64_t>(num_tokens) * p.shape.units_per_token;
  p.shape.part_chunks = static_cast<uint32_t>(part_elems / in);
  p.err = d_err;
  p.vec = in;
  p.prefetch = in >= 16 && on_device ? 1 : 0;
  p.scale_mode = scale_mode;
  p.scales_stride = scales_stride;
  return i64 ? launch_gather_fp8<int64_t>(in, fmt, bf16, p, stream)
             : launch_gather_fp8<int32_t>(in, fmt, bf16, p, stream);
}

}  // namespace

extern "C" kv_status kv_gather_fp8(const void* k_cache, const void* v_cache, void* k_out,
                                   void* v_out, const void* indices, kv_index_dtype index_dtype,
                                   int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                   int32_t head_dim, kv_src_dtype out_dtype, const kv_strides* s,
                                   int64_t page_size, int64_t kc_page_stride,
                                   int64_t vc_page_stride, int64_t size_limit,
                                   const float* k_scale, const float* v_scale, int32_t use_scale,
                                   kv_error_record* d_err, kv_stream_t stream) {
  return gather_fp8(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                    num_tokens, num_heads, head_dim, out_dtype, s, page_size, kc_page_stride,
                    vc_page_stride, size_limit, kFmtE4M3,
                    use_scale ? KV_SCALE_TENSOR : KV_SCALE_NONE, k_scale, v_scale, nullptr,
                    nullptr, 0, d_err, stream);
}

extern "C" kv_status kv_gather_fp8_ex(const void* k_cache, const void* v_cache, void* k_out,
                                      void* v_out, const void* indices, kv_index_dtype index_dtype,
                                      int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                      int32_t head_dim, kv_src_dtype out_dtype,
                                      const kv_strides* s, int64_t page_size,
                                      int64_t kc_page_stride, int64_t vc_page_stride,
                                      int64_t size_limit, kv_fp8_format format,
                                      kv_scale_mode scale_mode, const float* k_scale,
                                      const float* v_scale, const float* k_scales,
                                      const float* v_scales, int64_t scales_slot_stride,
                                      kv_error_record* d_err, kv_stream_t stream) {
  if (format != KV_FP8_E4M3FN && format != KV_FP8_E5M2) return KV_ERR_INVALID_ARG;
  if (scale_mode != KV_SCALE_NONE && scale_mode != KV_SCALE_TENSOR && scale_mode != KV_SCALE_TOKEN &&
      scale_mode != KV_SCALE_TOKEN_HEAD && scale_mode != KV_SCALE_PAGE)
    return KV_ERR_INVALID_ARG;
  return gather_fp8(k_cache, v_cache, k_out, v_out, indices, index_dtype, index_stride,
                    num_tokens, num_heads, head_dim, out_dtype, s, page_size, kc_page_stride,
                    vc_page_stride, size_limit, format == KV_FP8_E5M2 ? kFmtE5M2 : kFmtE4M3,
                    scale_mode, k_scale, v_scale, k_scales, v_scales, scales_slot_stride, d_err,
                    stream);
}
