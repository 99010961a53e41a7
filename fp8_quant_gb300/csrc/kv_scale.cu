// Scale preparation on the device, so that a captured step needs no host
// synchronisation (sglang trtllm_fp8_kv_kernel.py, `fused_fp8_set_kv_buffer`
// forms the inverse scales 1.0 / scale on the GPU for exactly that reason):
//
//   kv_inv_scale   inv[i] = 1 / scale[i], fp32, round to nearest;
//   kv_absmax_inv  per-tensor max |x| of the K rows and of the V rows (NaN
//                  ignored) and inv = fp8_max / amax (1 when amax is 0), the
//                  per-tensor inverse scale kv_store_fp8 consumes.
//
// The absmax pass is a pure HBM read stream.  A resident grid of a few CTAs
// per SM (half of each SM's warp slots, so that the next call's CTAs can
// become resident beside it): before the programmatic-launch wait every warp
// prefetches all of its rows into L2, its lanes in parallel; after it a warp
// keeps two rows' loads in flight, CTAs reduce their warps in shared memory,
// and one atomicMax per CTA and tensor lands on the float bits of an
// accumulator (for non-negative floats the bit patterns order like the
// values).  A one-CTA finish kernel then turns the accumulators into amax and
// inv.  With a caller workspace the finish also clears the accumulators for
// the next call (two launches); without one, a zeroing kernel runs first and
// the caller's amax output is the accumulator (three launches).
// Measured on GB300 (per-call time, back-to-back calls, 33.5 MB read): the
// reduction alone 5.9 us; with the workspace 7.1 us; the earlier three-launch
// chain 7.5 us.  A single launch whose last CTA finishes (an acquire-release
// completion counter) measured 7.1 us: that CTA's chain of dependent atomics
// costs more than a launch hand-over, and a 128-bit compare-and-swap carrying
// both maxima and the count serialised to 50-450 us.
#include "kv_host.h"

#ifndef KV_ABSMAX_CTAS_PER_SM
#define KV_ABSMAX_CTAS_PER_SM 4  // CTAs of KV_ABSMAX_THREADS per SM
#endif
#ifndef KV_ABSMAX_THREADS
#define KV_ABSMAX_THREADS 256
#endif
#ifndef KV_ABSMAX_ILP
#define KV_ABSMAX_ILP 2          // units whose loads a warp keeps in flight together
#endif
#ifndef KV_ABSMAX_FINISH_THREADS
#define KV_ABSMAX_FINISH_THREADS 32  // the one-CTA finish kernel (and the zeroing kernel)
#endif
#ifndef KV_ABSMAX_PREFETCH
#define KV_ABSMAX_PREFETCH 1     // L2 prefetch of all of a warp's units before the grid wait
#endif
static_assert(KV_ABSMAX_THREADS % 32 == 0 && KV_ABSMAX_THREADS <= kvimpl::kThreads, "CTA size");

namespace kvimpl {
namespace {

struct InvParams {
  const float* scale;
  float* inv;
  int64_t n;
};

__global__ void __launch_bounds__(kThreads) kv_inv_kernel(const __grid_constant__ InvParams p) {
  grid_handover<true>();  // small bookkeeping kernel: let the next kernel in early
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.n; i += stride)
    p.inv[i] = __fdiv_rn(1.0f, p.scale[i]);
}

struct AbsmaxParams {
  const uint8_t* src[2];
  int64_t token[2], seg[2];  // byte strides of the rows and of their segments
  UnitShape shape;           // units: (token, K|V, segment); parts = 1
  unsigned int* amax_bits;   // two accumulator words: K, V
  uint64_t* tagged;          // non-null: the tagged accumulators of the fused dynamic write instead
  int vec;                   // bytes per chunk
  int prefetch;              // rows are device memory with 16-byte aligned segments
};

// |x| of the two 2-byte elements in `w`, folded into m (fmaxf ignores NaN).
template <bool kBF16>
__device__ __forceinline__ float absmax2(float m, uint32_t w) {
  const float2 x = widen2<kBF16>(w);
  return fmaxf(m, fmaxf(fabsf(x.x), fabsf(x.y)));
}

__device__ __forceinline__ const uint8_t* absmax_row(const AbsmaxParams& p, const Unit& w) {
  return p.src[w.kv] + w.token * p.token[w.kv] + static_cast<int64_t>(w.seg) * p.seg[w.kv];
}

// Unit u of an absmax launch.  With one segment per row (heads contiguous)
// the unit is (token u / 2, side u % 2): shifts instead of the general
// decode's 64-bit division, which sits before every row's loads (measured:
// 7.47 -> 7.13 us per call on the fp8 batch).
__device__ __forceinline__ Unit absmax_unit(const AbsmaxParams& p, uint64_t u) {
  if (p.shape.units_per_token == 2) {
    Unit w;
    w.token = static_cast<int64_t>(u >> 1);
    w.kv = static_cast<uint32_t>(u & 1u);
    w.rank = w.kv;
    w.seg = 0;
    w.part = 0;
    return w;
  }
  return decode_unit(p.shape, u);
}

// One warp per (token, K|V, segment) unit, ILP units at a time (units u,
// u + nwarps, ...); a lane issues up to U vector loads of each of them before
// it reduces, so a warp keeps 32*U*VEC*ILP bytes in flight.
template <int VEC, int U, int ILP, bool kBF16>
__global__ void __launch_bounds__(kThreads) kv_absmax_rows(const __grid_constant__ AbsmaxParams p) {
  __shared__ float part[2][kMaxWarpsPerCta];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t warp = threadIdx.x >> 5;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  const uint64_t first = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + warp;
  const uint32_t nchunks = p.shape.part_chunks;
  if (KV_ABSMAX_PREFETCH && p.prefetch) {  // every unit this warp will read, lanes in parallel
    for (uint64_t u = first + lane * nwarps; u < p.shape.num_units; u += 32u * nwarps)
      prefetch_l2_bulk(absmax_row(p, absmax_unit(p, u)),
                       nchunks * static_cast<uint32_t>(p.vec));
  }
  grid_handover();
  float m0 = 0.0f, m1 = 0.0f;
  for (uint64_t u = first; u < p.shape.num_units; u += nwarps * ILP) {
    const uint8_t* src[ILP];
    uint32_t side[ILP];
    float acc[ILP];
#pragma unroll
    for (int i = 0; i < ILP; ++i) {
      const uint64_t ui = u + i * nwarps;
      acc[i] = 0.0f;
      side[i] = 0;
      src[i] = nullptr;
      if (ui < p.shape.num_units) {
        const Unit w = absmax_unit(p, ui);
        src[i] = absmax_row(p, w);
        side[i] = w.kv;
      }
    }
    for (uint32_t c0 = 0; c0 < nchunks; c0 += 32u * U) {
      Chunk<VEC> ch[ILP][U];
#pragma unroll
      for (int i = 0; i < ILP; ++i)
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const uint32_t c = c0 + lane + 32u * j;
          if (src[i] != nullptr && c < nchunks) ld_stream(ch[i][j], src[i] + static_cast<size_t>(c) * VEC);
        }
#pragma unroll
      for (int i = 0; i < ILP; ++i)
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const uint32_t c = c0 + lane + 32u * j;
          if (src[i] == nullptr || c >= nchunks) continue;
          if constexpr (VEC >= 4) {
#if KV_PACKED_MATH
            uint32_t pm = 0;
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) pm = absmax_pair<kBF16>(pm, ch[i][j].w[q]);
            acc[i] = fmaxf(acc[i], absmax_pair_value<kBF16>(pm));
#else
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q) acc[i] = absmax2<kBF16>(acc[i], ch[i][j].w[q]);
#endif
          } else {
            acc[i] = absmax2<kBF16>(acc[i], static_cast<uint32_t>(ch[i][j].h));  // upper element is 0
          }
        }
    }
#pragma unroll
    for (int i = 0; i < ILP; ++i) {
      if (side[i]) m1 = fmaxf(m1, acc[i]);
      else m0 = fmaxf(m0, acc[i]);
    }
  }
  float m[2] = {m0, m1};
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    m[kv] = warp_absmax(m[kv]);
    if (lane == 0) part[kv][warp] = m[kv];
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    float v = 0.0f;
#pragma unroll
    for (uint32_t i = 0; i < warps_per_cta(); ++i) v = fmaxf(v, part[threadIdx.x][i]);
    if (p.tagged != nullptr) {
      // (generation << 16) | the maximum's 16-bit pattern (exact: a maximum of
      // 16-bit inputs is one of them; non-negative patterns order like their
      // values), so a later call's words always win: nothing is cleared
      const uint64_t gen = p.tagged[0];
      const uint32_t bits = kBF16 ? (__float_as_uint(v) >> 16)
                                  : static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v)));
      atomicMax(reinterpret_cast<unsigned long long*>(p.tagged + 1 + threadIdx.x),
                static_cast<unsigned long long>((gen << 16) | bits));
    } else if (v > 0.0f) {
      atomicMax(p.amax_bits + threadIdx.x, __float_as_uint(v));
    }
  }
}

// Clears the two accumulator words.  A kernel rather than a memset so that
// zeroing, reduction and finish chain by programmatic launch.
__global__ void __launch_bounds__(kThreads) kv_absmax_zero(const __grid_constant__ AbsmaxParams p) {
  grid_handover<true>();  // small bookkeeping kernel: let the next kernel in early
  if (blockIdx.x == 0 && threadIdx.x < 2) p.amax_bits[threadIdx.x] = 0u;
}

struct FinishParams {
  unsigned int* acc;   // the two accumulator words
  float* amax;
  float* inv;
  float fp8_max;
  int clear;           // clear the accumulators (a workspace) after reading them
};

__global__ void __launch_bounds__(kThreads) kv_absmax_finish(const __grid_constant__ FinishParams p) {
  grid_handover<true>();  // small bookkeeping kernel: let the next kernel in early
  if (threadIdx.x < 2) {
    const float a = __uint_as_float(p.acc[threadIdx.x]);
    if (p.clear) p.acc[threadIdx.x] = 0u;
    p.amax[threadIdx.x] = a;
    p.inv[threadIdx.x] = a > 0.0f ? __fdiv_rn(p.fp8_max, a) : 1.0f;
  }
}

template <int VEC>
kv_status launch_absmax(bool bf16, const AbsmaxParams& p, cudaStream_t stream, uint64_t max_ctas) {
  constexpr int U = VEC == 32 ? 2 : 4;
  constexpr int ILP = KV_ABSMAX_ILP;
  const uint64_t warps = (p.shape.num_units + ILP - 1) / ILP;
  if (bf16)
    return launch(kv_absmax_rows<VEC, U, ILP, true>, warps, p, stream, max_ctas, KV_ABSMAX_THREADS);
  return launch(kv_absmax_rows<VEC, U, ILP, false>, warps, p, stream, max_ctas, KV_ABSMAX_THREADS);
}

}  // namespace
}  // namespace kvimpl

using namespace kvimpl;

extern "C" kv_status kv_inv_scale(const float* scale, float* inv, int64_t n, kv_stream_t stream_) {
  if (n < 0) return KV_ERR_INVALID_ARG;
  if (n == 0) return KV_OK;
  if (!scale || !inv || ((u64(scale) | u64(inv)) & 3u) != 0) return KV_ERR_INVALID_ARG;
  // one thread per value: as many warps as 32-value groups
  return launch(kv_inv_kernel, (static_cast<uint64_t>(n) + 31) / 32, InvParams{scale, inv, n},
                reinterpret_cast<cudaStream_t>(stream_));
}

// The reduction launch shared by kv_absmax_inv and the fused dynamic
// per-tensor write: acc (two 32-bit words, float bits) or tagged (the fused
// write's workspace).  Arguments are checked by the callers; num_tokens > 0.
kv_status kvimpl::absmax_reduce(const void* k, const void* v, kv_src_dtype src_dtype,
                                int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                                const kv_strides* s, unsigned int* acc, uint64_t* tagged,
                                bool on_device, cudaStream_t stream) {
  const int64_t head_bytes = 2 * static_cast<int64_t>(head_dim);
  const bool merged = num_heads == 1 || (s->k_head == head_bytes && s->v_head == head_bytes);
  const uint32_t nseg = merged ? 1u : static_cast<uint32_t>(num_heads);
  const int64_t seg_bytes = merged ? head_bytes * num_heads : head_bytes;
  uint64_t bits = u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token) | u64(seg_bytes);
  if (!merged) bits |= u64(s->k_head) | u64(s->v_head);
  const int vec = pow2_align(bits);
  AbsmaxParams p = {};
  p.src[0] = static_cast<const uint8_t*>(k);
  p.src[1] = static_cast<const uint8_t*>(v);
  p.token[0] = s->k_token;
  p.token[1] = s->v_token;
  p.seg[0] = s->k_head;
  p.seg[1] = s->v_head;
  p.shape.parts = 1;
  p.shape.units_per_side = nseg;
  p.shape.units_per_token = 2u * nseg;
  p.shape.num_units = static_cast<uint64_t>(num_tokens) * p.shape.units_per_token;
  p.shape.part_chunks = static_cast<uint32_t>(seg_bytes / vec);
  p.amax_bits = acc;
  p.tagged = tagged;
  p.vec = vec;
  p.prefetch = vec >= 16 && on_device ? 1 : 0;
  // a resident grid of a few CTAs per SM loops over the rows, so only a few
  // hundred same-address atomics land at the end
  int sms = 0;
  const kv_status st = current_sm_count(&sms);
  if (st != KV_OK) return st;
  const uint64_t max_ctas = static_cast<uint64_t>(sms) * KV_ABSMAX_CTAS_PER_SM;
  const bool bf16 = src_dtype == KV_SRC_BF16;
  switch (vec) {
#if KV_MAX_VEC >= 32
    case 32: return launch_absmax<32>(bf16, p, stream, max_ctas);
#endif
    case 16: return launch_absmax<16>(bf16, p, stream, max_ctas);
    case 8: return launch_absmax<8>(bf16, p, stream, max_ctas);
    case 4: return launch_absmax<4>(bf16, p, stream, max_ctas);
    default: return launch_absmax<2>(bf16, p, stream, max_ctas);
  }
}

extern "C" kv_status kv_absmax_inv(const void* k, const void* v, kv_src_dtype src_dtype,
                                   int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                                   const kv_strides* s, float fp8_max, float* amax, float* inv,
                                   uint32_t* work, kv_stream_t stream_) {
  if (num_tokens < 0 || num_heads < 1 || head_dim < 1) return KV_ERR_INVALID_ARG;
  if (!s || !amax || !inv || ((u64(amax) | u64(inv) | u64(work)) & 3u) != 0)
    return KV_ERR_INVALID_ARG;
  if (num_tokens > 0 && (!k || !v)) return KV_ERR_INVALID_ARG;
  if (src_dtype != KV_SRC_F16 && src_dtype != KV_SRC_BF16) return KV_ERR_INVALID_ARG;
  if (!(fp8_max > 0.0f) || fp8_max == INFINITY) return KV_ERR_INVALID_ARG;
  if (s->k_dim != 2 || s->v_dim != 2) return KV_ERR_UNSUPPORTED;
  if (((u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token) | u64(s->k_head) | u64(s->v_head)) & 1u) != 0)
    return KV_ERR_INVALID_ARG;
  if (num_tokens > (int64_t{1} << 40)) return KV_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  bool on_device = true;
  if (num_tokens > 0) {
    const void* in[4] = {k, v, amax, inv};
    const kv_status cs = classify_inputs(in, 4, &on_device);
    if (cs != KV_OK) return cs;
  }
  // Accumulators: the caller's workspace (zero on entry, cleared again by the
  // finish), else the amax output, zeroed by a kernel first.
  unsigned int* acc = work != nullptr ? reinterpret_cast<unsigned int*>(work)
                                      : reinterpret_cast<unsigned int*>(amax);
  kv_status st = KV_OK;
  if (work == nullptr) {
    AbsmaxParams zp = {};
    zp.amax_bits = acc;
    st = launch(kv_absmax_zero, 1, zp, stream, 0, KV_ABSMAX_FINISH_THREADS);
    if (st != KV_OK) return st;
  }
  if (num_tokens > 0) {
    st = absmax_reduce(k, v, src_dtype, num_tokens, num_heads, head_dim, s, acc, nullptr, on_device,
                       stream);
    if (st != KV_OK) return st;
  }
  return launch(kv_absmax_finish, 1, FinishParams{acc, amax, inv, fp8_max, work != nullptr ? 1 : 0},
                stream, 0, KV_ABSMAX_FINISH_THREADS);
}
