// Extended FP8 write: e4m3fn or e5m2 caches, and dynamic scales computed in
// the kernel per token row or per (token, head).
//
// The fused FP8 write's module docstring (sglang trtllm_fp8_kv_kernel.py)
// names "per-token or per-page scale computation" but its kernel only takes
// a per-tensor scale; this file supplies the per-token form.  For each group
// (the K or V row of a token, or one head of it): amax = max |x| (NaN
// ignored); inv = fmax / amax and scale = amax / fmax in fp32 (both 1 when
// amax is 0); codes = fp8(x * inv); `scale` goes to the caller's per-slot
// scale cache.  fmax is 448 for e4m3fn and 57344 for e5m2.
//
// One warp owns one group.  The group's elements are loaded once into
// registers (up to 4 chunks per lane, 2 for 16-byte chunks; longer groups
// are re-read from L2 in a second pass), the warp reduces amax with shuffles, then converts and stores
// the codes and lane 0 stores the group's scale.  As in the other write
// kernels, the group's source bytes are prefetched into L2 before the
// programmatic-launch wait.
#include "kv_host.h"

#ifndef KV_DYN_STAGED
#define KV_DYN_STAGED 1              // staged (shared-memory ring) form of the row-layout write
#endif
#ifndef KV_DYN_CONSUMERS
#define KV_DYN_CONSUMERS 8           // consumer warps per CTA of the staged form
#endif
#ifndef KV_DYN_CTAS_PER_SM
#define KV_DYN_CTAS_PER_SM 2
#endif
#ifndef KV_DYN_STAGE_BYTES
#define KV_DYN_STAGE_BYTES (96 * 1024)  // shared memory for the stages of one CTA
#endif

namespace kvimpl {
namespace {

constexpr uint32_t kDynMaxStages = 64;

struct DynSide {
  const uint8_t* src;
  uint8_t* dst;
  int64_t src_token, src_seg;              // input byte strides (segment = head)
  int64_t dst_slot, dst_seg, dst_page;     // cache byte strides
  float* scales;                           // per-slot scale cache
};

struct DynParams {
  DynSide side[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size, scales_stride;
  uint64_t num_units;  // num_tokens * 2 * groups
  uint32_t groups;     // groups per row: 1 (token) or num_heads (token, head)
  uint32_t gseg;       // segments per group
  uint32_t cps;        // chunks per segment
  float fmax;
  kv_error_record* err;
  int prefetch;        // segments 16-byte aligned: bulk L2 prefetch allowed
};

struct DynUnit {
  int64_t token;
  uint32_t kv, group, rank;
};

__device__ __forceinline__ DynUnit dyn_unit(const DynParams& p, uint64_t u) {
  DynUnit w;
  const uint64_t per_token = 2ull * p.groups;
  const uint64_t t = u / per_token;
  w.token = static_cast<int64_t>(t);
  w.rank = static_cast<uint32_t>(u - t * per_token);
  w.kv = w.rank >= p.groups ? 1u : 0u;
  w.group = w.rank - w.kv * p.groups;
  return w;
}

// amax of the CH elements of one input chunk, folded into m.
template <int CH, bool kBF16>
__device__ __forceinline__ float chunk_absmax(float m, const Chunk<2 * CH>& c) {
  if constexpr (CH >= 2) {
#pragma unroll
    for (int i = 0; i < CH / 2; ++i) {
      const float2 x = widen2<kBF16>(c.w[i]);
      m = fmaxf(m, fmaxf(fabsf(x.x), fabsf(x.y)));
    }
  } else {
    const float2 x = widen2<kBF16>(static_cast<uint32_t>(c.h));
    m = fmaxf(m, fabsf(x.x));
  }
  return m;
}

// CH codes of one chunk.
template <int CH, bool kBF16, int FMT>
__device__ __forceinline__ Chunk<CH> chunk_quant(const Chunk<2 * CH>& c, float inv) {
  Chunk<CH> o;
  if constexpr (CH >= 4) {
#pragma unroll
    for (int i = 0; i < CH / 4; ++i)
      o.w[i] = quant2<kBF16, FMT>(c.w[2 * i], inv) | (quant2<kBF16, FMT>(c.w[2 * i + 1], inv) << 16);
  } else if constexpr (CH == 2) {
    o.h = static_cast<uint16_t>(quant2<kBF16, FMT>(c.w[0], inv));
  } else {
    o.h = static_cast<uint16_t>(quant2<kBF16, FMT>(static_cast<uint32_t>(c.h), inv) & 0xFFu);
  }
  return o;
}

template <int CH, typename IdxT, bool kBF16, int FMT>
__global__ void __launch_bounds__(kThreads) kv_fp8_dyn_rows(const __grid_constant__ DynParams p) {
  constexpr int kMaxJ = CH >= 8 ? 2 : 4;  // chunks per lane held in registers (16-byte chunks: 2, no spill)
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
  const uint32_t n = p.gseg * p.cps;  // chunks in a group
  const int64_t seg_in = static_cast<int64_t>(p.cps) * CH * 2;

  if (KV_PREFETCH && p.prefetch && u < p.num_units) {
    const DynUnit w = dyn_unit(p, u);
    const DynSide& sd = p.side[w.kv];
    const uint8_t* base = sd.src + w.token * sd.src_token +
                          static_cast<int64_t>(w.group) * p.gseg * sd.src_seg;
    for (uint32_t sg = lane; sg < p.gseg; sg += 32u)
      prefetch_l2_bulk(base + static_cast<int64_t>(sg) * sd.src_seg, static_cast<uint32_t>(seg_in));
    if (lane == 0) prefetch_l2_line(static_cast<const IdxT*>(p.indices) + w.token * p.index_stride);
  }
  grid_handover();

  for (; u < p.num_units; u += nwarps) {
    const DynUnit w = dyn_unit(p, u);
    const DynSide& sd = p.side[w.kv];
    const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, w.token);
    const uint8_t* src = sd.src + w.token * sd.src_token +
                         static_cast<int64_t>(w.group) * p.gseg * sd.src_seg;
    auto src_of = [&](uint32_t c) {
      const uint32_t sg = c / p.cps;
      return src + static_cast<int64_t>(sg) * sd.src_seg + static_cast<int64_t>(c - sg * p.cps) * (2 * CH);
    };
    const bool in_regs = n <= 32u * kMaxJ;
    Chunk<2 * CH> buf[kMaxJ];
    float amax = 0.0f;
    if (in_regs) {
#pragma unroll
      for (int j = 0; j < kMaxJ; ++j) {
        const uint32_t c = lane + 32u * j;
        if (c < n) ld_stream(buf[j], src_of(c));
      }
#pragma unroll
      for (int j = 0; j < kMaxJ; ++j)
        if (lane + 32u * j < n) amax = chunk_absmax<CH, kBF16>(amax, buf[j]);
    } else {
      for (uint32_t c = lane; c < n; c += 32u) {
        Chunk<2 * CH> t;
        ld_stream(t, src_of(c));
        amax = chunk_absmax<CH, kBF16>(amax, t);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if (slot < 0 || slot >= p.size_limit) {
      if (w.rank == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(w.token));
      continue;
    }
    const bool pos = amax > 0.0f;
    const float inv = pos ? __fdiv_rn(p.fmax, amax) : 1.0f;
    uint8_t* dst = sd.dst + paged_offset(slot, p.page_size, sd.dst_page, sd.dst_slot) +
                   static_cast<int64_t>(w.group) * p.gseg * sd.dst_seg;
    auto dst_of = [&](uint32_t c) {
      const uint32_t sg = c / p.cps;
      return dst + static_cast<int64_t>(sg) * sd.dst_seg + static_cast<int64_t>(c - sg * p.cps) * CH;
    };
    if (in_regs) {
#pragma unroll
      for (int j = 0; j < kMaxJ; ++j) {
        const uint32_t c = lane + 32u * j;
        if (c < n) st_stream(dst_of(c), chunk_quant<CH, kBF16, FMT>(buf[j], inv));
      }
    } else {
      for (uint32_t c = lane; c < n; c += 32u) {
        Chunk<2 * CH> t;
        ld_stream(t, src_of(c));
        st_stream(dst_of(c), chunk_quant<CH, kBF16, FMT>(t, inv));
      }
    }
    if (lane == 0)
      sd.scales[slot * p.scales_stride + w.group] = pos ? __fdiv_rn(amax, p.fmax) : 1.0f;
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// Fast path for rows whose heads are contiguous on both sides: the layout of
// the static FP8 write (lane l converts the 16-element chunks l, l+32, ... of
// a row: 32 input bytes, 16 output bytes each), with each group's amax
// reduced over the lanes that hold it.  A head of D elements is D/16
// consecutive chunks, so in every 32-chunk slab of the row it sits on an
// aligned run of D/16 lanes; a shuffle over those lanes gives its amax.  In
// the per-token mode the group is the whole row.  Large launches pair the K
// and the V row of a token in one warp (NS == 2).
struct DynRowParams {
  DynSide side[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size, scales_stride;
  UnitShape shape;          // units: (token, K|V) rows, or tokens when paired
  uint32_t chunks;          // 16-element chunks per row
  uint32_t group_chunks;    // chunks per scale group (D / 16), or 0: the whole row
  float fmax;
  kv_error_record* err;
  int prefetch;             // rows in device memory: bulk L2 prefetch allowed
};

template <int J, int NS, typename IdxT, bool kBF16, int FMT>
__global__ void __launch_bounds__(kThreads) kv_fp8_dyn_row(const __grid_constant__ DynRowParams p) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
  const uint32_t n = p.chunks;
  const uint32_t g = p.group_chunks;
  if (KV_PREFETCH && p.prefetch && lane == 0 && u < p.shape.num_units) {
    const Unit w = decode_unit(p.shape, u);
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const DynSide& sd = p.side[NS == 2 ? i : w.kv];
      prefetch_l2_bulk(sd.src + w.token * sd.src_token, n * 32u);
    }
    prefetch_l2_line(static_cast<const IdxT*>(p.indices) + w.token * p.index_stride);
  }
  grid_handover();

  for (; u < p.shape.num_units; u += nwarps) {
    const Unit w = decode_unit(p.shape, u);
    const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, w.token);
    Chunk<32> buf[NS][J];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const DynSide& sd = p.side[NS == 2 ? i : w.kv];
      const uint8_t* src = sd.src + w.token * sd.src_token;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const uint32_t c = lane + 32u * j;
        if (c < n) ld_stream(buf[i][j], src + static_cast<size_t>(c) * 32u);
      }
    }
    float a[NS][J];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
#pragma unroll
      for (int j = 0; j < J; ++j)
        a[i][j] = lane + 32u * j < n ? chunk_absmax<16, kBF16>(0.0f, buf[i][j]) : 0.0f;
      if (g != 0) {             // per head: the aligned run of g lanes
        for (uint32_t o = 1; o < g; o <<= 1)
#pragma unroll
          for (int j = 0; j < J; ++j) a[i][j] = fmaxf(a[i][j], __shfl_xor_sync(0xFFFFFFFFu, a[i][j], o));
      } else {                  // per token: the whole row
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < J; ++j) m = fmaxf(m, a[i][j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
#pragma unroll
        for (int j = 0; j < J; ++j) a[i][j] = m;
      }
    }
    if (slot < 0 || slot >= p.size_limit) {
      if (w.rank == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(w.token));
      continue;
    }
    // The warp holds NS * gps groups (gps per row).  Lane k computes the
    // two divisions of group k, once: its amax comes from the lane holding
    // the group's first chunk, and every lane then takes the inverse scale
    // of its chunks' groups from lane k.
    const uint32_t gps = g != 0 ? n / g : 1u;
    const uint32_t gk = lane % gps;                       // lane's group within its side
    const uint32_t c0 = g != 0 ? gk * g : 0u;             // first chunk of that group
    float amax_k = 0.0f;
#pragma unroll
    for (int i = 0; i < NS; ++i)
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float v = __shfl_sync(0xFFFFFFFFu, a[i][j], c0 % 32u);
        if (lane / gps == static_cast<uint32_t>(i) && c0 / 32u == static_cast<uint32_t>(j)) amax_k = v;
      }
    const bool pos_k = amax_k > 0.0f;
    const bool owner = lane < NS * gps;
    const float inv_k = owner && pos_k ? __fdiv_rn(p.fmax, amax_k) : 1.0f;
    if (owner) {
      const DynSide& sd = p.side[NS == 2 ? lane / gps : w.kv];
      sd.scales[slot * p.scales_stride + gk] = pos_k ? __fdiv_rn(amax_k, p.fmax) : 1.0f;
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const DynSide& sd = p.side[NS == 2 ? i : w.kv];
      uint8_t* dst = sd.dst + paged_offset(slot, p.page_size, sd.dst_page, sd.dst_slot);
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const uint32_t c = lane + 32u * j;
        const uint32_t k = static_cast<uint32_t>(i) * gps + (g != 0 ? c / g : 0u);
        const float inv = __shfl_sync(0xFFFFFFFFu, inv_k, k < 32u ? k : 0u);
        if (c < n) st_stream(dst + static_cast<size_t>(c) * 16u, chunk_quant<16, kBF16, FMT>(buf[i][j], inv));
      }
    }
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

template <int J, typename IdxT, int FMT>
kv_status launch_dyn_row_j(bool bf16, const DynRowParams& p, cudaStream_t stream) {
  if (p.shape.num_units >= KV_LARGE_LAUNCH_WARPS) {
    DynRowParams q = p;   // one warp per token: K and V rows together
    q.shape.units_per_token = 1;
    q.shape.units_per_side = 1;
    q.shape.num_units /= 2;
    if (bf16) return launch(kv_fp8_dyn_row<J, 2, IdxT, true, FMT>, q.shape.num_units, q, stream);
    return launch(kv_fp8_dyn_row<J, 2, IdxT, false, FMT>, q.shape.num_units, q, stream);
  }
  if (bf16) return launch(kv_fp8_dyn_row<J, 1, IdxT, true, FMT>, p.shape.num_units, p, stream);
  return launch(kv_fp8_dyn_row<J, 1, IdxT, false, FMT>, p.shape.num_units, p, stream);
}

template <typename IdxT, int FMT>
kv_status launch_dyn_row_fmt(int j, bool bf16, const DynRowParams& p, cudaStream_t stream) {
  if (j == 1) return launch_dyn_row_j<1, IdxT, FMT>(bf16, p, stream);
  if (j == 2) return launch_dyn_row_j<2, IdxT, FMT>(bf16, p, stream);
  return launch_dyn_row_j<4, IdxT, FMT>(bf16, p, stream);
}

template <typename IdxT>
kv_status launch_dyn_row(int j, int fmt, bool bf16, const DynRowParams& p, cudaStream_t stream) {
  if (fmt == kFmtE5M2) return launch_dyn_row_fmt<IdxT, kFmtE5M2>(j, bf16, p, stream);
  return launch_dyn_row_fmt<IdxT, kFmtE4M3>(j, bf16, p, stream);
}

// ---------------------------------------------------------------------------
// Staged form of the row-layout dynamic write (device-resident inputs, rows a
// multiple of 512 bytes).  The whole row must be in hand before any code can
// be formed, and a warp that holds its rows in registers has nothing to do
// while they arrive.  Here one producer thread per CTA streams the K and V
// rows of the CTA's tokens into a ring of shared-memory stages with bulk
// asynchronous copies (one mbarrier per stage carries the byte count), so the
// loads of later tokens are in flight while consumer warps reduce, convert
// and store earlier ones; a consumer frees its stage by arriving on the
// stage's second mbarrier.  Lane l of a consumer takes the 16-byte pieces l,
// l+32, ... of each row: a scale group (a head of D elements: D/8 pieces, or
// the whole row) is an aligned run of lanes in one 32-piece slab, or whole
// slabs.  Every wait is bounded; a wait that gives up sets the timeout bit of
// the error record, and the CTA then waits (bounded) for the copies it
// issued before it exits.
// ---------------------------------------------------------------------------
struct StagedParams {
  DynSide side[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size, scales_stride;
  int64_t num_tokens;
  uint32_t row_bytes;     // R: a multiple of 512
  uint32_t group_pieces;  // 16-byte pieces per scale group: D / 8, or R / 16 (whole row)
  uint32_t stages;        // ring depth (each stage holds one token's K and V rows)
  float fmax;
  kv_error_record* err;
  int prefetch;           // L2 prefetch of the first tokens before the grid wait
};

template <int P, typename IdxT, bool kBF16, int FMT>  // P: pieces per lane and row (R / 512)
__global__ void __launch_bounds__(32 * (KV_DYN_CONSUMERS + 1))
    kv_fp8_dyn_staged(const __grid_constant__ StagedParams p) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ uint32_t issued[kDynMaxStages];  // copies issued per stage
  __shared__ int aborted;
  const uint32_t S = p.stages;
  const uint32_t R = p.row_bytes;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint64_t G = gridDim.x;
  const int64_t nk = p.num_tokens > static_cast<int64_t>(blockIdx.x)
                         ? (p.num_tokens - 1 - static_cast<int64_t>(blockIdx.x)) / static_cast<int64_t>(G) + 1
                         : 0;  // tokens of this CTA: blockIdx.x + k * G
  const uint32_t data0 = smem_addr(stage_mem);
  const uint32_t full0 = data0 + S * 2u * R;  // full[s]: the stage's rows have landed
  const uint32_t empty0 = full0 + 8u * S;     // empty[s]: its consumer is done with it
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
      issued[s] = 0;
    }
    aborted = 0;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // inits seen by the copy engine
  }
  if (KV_PREFETCH && p.prefetch && warp == 0) {
    for (int64_t k = lane; k < nk && k < static_cast<int64_t>(S); k += 32) {
      const int64_t t = static_cast<int64_t>(blockIdx.x) + k * static_cast<int64_t>(G);
      prefetch_l2_bulk(p.side[0].src + t * p.side[0].src_token, R);
      prefetch_l2_bulk(p.side[1].src + t * p.side[1].src_token, R);
    }
  }
  __syncthreads();
  grid_handover();

  if (warp == 0) {
    if (lane == 0) {  // producer
      for (int64_t k = 0; k < nk; ++k) {
        const uint32_t s = static_cast<uint32_t>(k % S);
        const uint32_t n = static_cast<uint32_t>(k / S);
        if (n > 0 && !mbar_wait(empty0 + 8u * s, (n - 1u) & 1u)) {
          record_timeout(p.err);
          atomicExch(&aborted, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&aborted)) break;
        const int64_t t = static_cast<int64_t>(blockIdx.x) + k * static_cast<int64_t>(G);
        const uint32_t buf = data0 + s * 2u * R;
        mbar_expect_tx(full0 + 8u * s, 2u * R);
        bulk_load(buf, p.side[0].src + t * p.side[0].src_token, R, full0 + 8u * s);
        bulk_load(buf + R, p.side[1].src + t * p.side[1].src_token, R, full0 + 8u * s);
        issued[s] = n + 1u;
      }
    }
  } else {  // consumers
    const uint32_t gp = p.group_pieces;
    const uint32_t gpr = 32u * P / gp;        // scale groups per row
    const uint32_t my_g = lane < 2u * gpr ? lane : 0u;  // the group this lane divides for
    const uint32_t my_i = my_g / gpr;                   // its side
    const uint32_t my_q0 = (my_g - my_i * gpr) * gp;    // its first piece
    for (int64_t k = warp - 1; k < nk; k += KV_DYN_CONSUMERS) {
      const uint32_t s = static_cast<uint32_t>(k % S);
      const uint32_t n = static_cast<uint32_t>(k / S);
      const int64_t t = static_cast<int64_t>(blockIdx.x) + k * static_cast<int64_t>(G);
      const int64_t slot = load_slot<IdxT>(p.indices, p.index_stride, t);
      if (!mbar_wait(full0 + 8u * s, n & 1u)) {
        if (lane == 0) {
          record_timeout(p.err);
          atomicExch(&aborted, 1);
        }
        break;
      }
      const uint32_t buf = data0 + s * 2u * R;
      uint32_t x[2][P][4];
      float a[2][P];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < P; ++j) {
          lds16(x[i][j], buf + static_cast<uint32_t>(i) * R + (lane + 32u * j) * 16u);
          float m = 0.0f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float2 v = widen2<kBF16>(x[i][j][w]);
            m = fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y)));
          }
          a[i][j] = m;
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * s);  // the rows are in registers: free the stage
      // group maxima: a run of gp lanes inside a slab, or whole slabs
      if (gp < 32u) {
        for (uint32_t o = 1; o < gp; o <<= 1)
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < P; ++j) a[i][j] = fmaxf(a[i][j], __shfl_xor_sync(0xFFFFFFFFu, a[i][j], o));
      } else {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < P; ++j)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a[i][j] = fmaxf(a[i][j], __shfl_xor_sync(0xFFFFFFFFu, a[i][j], o));
        const uint32_t slabs = gp / 32u;  // slabs per group (a power of two dividing P)
#pragma unroll
        for (int e = 1; e < P; e <<= 1) {  // xor steps stay inside aligned blocks of `slabs`
          if (static_cast<uint32_t>(e) >= slabs) break;
          float b[2][P];
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < P; ++j) b[i][j] = fmaxf(a[i][j], a[i][j ^ e]);
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < P; ++j) a[i][j] = b[i][j];
        }
      }
      // lane g divides for group g: its maximum sits in slab my_q0 / 32 at lane my_q0 % 32
      float amax_g = 0.0f;
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const float v = __shfl_sync(0xFFFFFFFFu, a[i][j], my_q0 % 32u);
          if (my_i == static_cast<uint32_t>(i) && my_q0 / 32u == static_cast<uint32_t>(j)) amax_g = v;
        }
      const bool pos = amax_g > 0.0f;
      const float inv_g = pos ? __fdiv_rn(p.fmax, amax_g) : 1.0f;
      if (slot < 0 || slot >= p.size_limit) {
        if (lane == 0) record_oob(p.err, static_cast<uint64_t>(t));
        continue;
      }
      if (lane < 2u * gpr)
        p.side[my_i].scales[slot * p.scales_stride + (my_g - my_i * gpr)] =
            pos ? __fdiv_rn(amax_g, p.fmax) : 1.0f;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const DynSide& sd = p.side[i];
        uint8_t* dst = sd.dst + paged_offset(slot, p.page_size, sd.dst_page, sd.dst_slot);
#pragma unroll
        for (int j = 0; j < P; ++j) {
          const uint32_t q = lane + 32u * j;
          const float inv = __shfl_sync(0xFFFFFFFFu, inv_g, static_cast<uint32_t>(i) * gpr + q / gp);
          Chunk<8> o;
          o.w[0] = quant2<kBF16, FMT>(x[i][j][0], inv) | (quant2<kBF16, FMT>(x[i][j][1], inv) << 16);
          o.w[1] = quant2<kBF16, FMT>(x[i][j][2], inv) | (quant2<kBF16, FMT>(x[i][j][3], inv) << 16);
          st_stream(dst + static_cast<size_t>(q) * 8u, o);
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && aborted) {
    // a wait gave up: do not exit while a copy into this CTA's shared memory
    // may still be in flight (bounded as well)
    for (uint32_t s = 0; s < S; ++s)
      if (issued[s] > 0) (void)mbar_wait(full0 + 8u * s, (issued[s] - 1u) & 1u);
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

template <int P, typename IdxT, int FMT>
kv_status launch_dyn_staged_p(bool bf16, const StagedParams& p, cudaStream_t stream) {
  void (*kernel)(StagedParams) = bf16 ? kv_fp8_dyn_staged<P, IdxT, true, FMT>
                                      : kv_fp8_dyn_staged<P, IdxT, false, FMT>;
  const size_t smem = static_cast<size_t>(p.stages) * 2u * p.row_bytes + 16u * p.stages;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e);
  int sms = 0;
  kv_status st = current_sm_count(&sms);
  if (st != KV_OK) return st;
  int64_t grid = static_cast<int64_t>(sms) * KV_DYN_CTAS_PER_SM;
  if (grid > p.num_tokens) grid = p.num_tokens;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(32u * (KV_DYN_CONSUMERS + 1), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e != cudaSuccess) return cuda_fail(e);
  return KV_OK;
}

template <typename IdxT, int FMT>
kv_status launch_dyn_staged_fmt(int pieces, bool bf16, const StagedParams& p, cudaStream_t stream) {
  switch (pieces) {
    case 1: return launch_dyn_staged_p<1, IdxT, FMT>(bf16, p, stream);
    case 2: return launch_dyn_staged_p<2, IdxT, FMT>(bf16, p, stream);
    default: return launch_dyn_staged_p<4, IdxT, FMT>(bf16, p, stream);
  }
}

template <typename IdxT>
kv_status launch_dyn_staged(int pieces, int fmt, bool bf16, const StagedParams& p, cudaStream_t stream) {
  if (fmt == kFmtE5M2) return launch_dyn_staged_fmt<IdxT, kFmtE5M2>(pieces, bf16, p, stream);
  return launch_dyn_staged_fmt<IdxT, kFmtE4M3>(pieces, bf16, p, stream);
}

template <int CH, typename IdxT, int FMT>
kv_status launch_dyn_fmt(bool bf16, const DynParams& p, cudaStream_t stream) {
  if (bf16) return launch(kv_fp8_dyn_rows<CH, IdxT, true, FMT>, p.num_units, p, stream);
  return launch(kv_fp8_dyn_rows<CH, IdxT, false, FMT>, p.num_units, p, stream);
}

template <int CH, typename IdxT>
kv_status launch_dyn_ch(int fmt, bool bf16, const DynParams& p, cudaStream_t stream) {
  if (fmt == kFmtE5M2) return launch_dyn_fmt<CH, IdxT, kFmtE5M2>(bf16, p, stream);
  return launch_dyn_fmt<CH, IdxT, kFmtE4M3>(bf16, p, stream);
}

template <typename IdxT>
kv_status launch_dyn(int ch, int fmt, bool bf16, const DynParams& p, cudaStream_t stream) {
  switch (ch) {
    case 8: return launch_dyn_ch<8, IdxT>(fmt, bf16, p, stream);
    case 4: return launch_dyn_ch<4, IdxT>(fmt, bf16, p, stream);
    case 2: return launch_dyn_ch<2, IdxT>(fmt, bf16, p, stream);
    default: return launch_dyn_ch<1, IdxT>(fmt, bf16, p, stream);
  }
}

}  // namespace
}  // namespace kvimpl

using namespace kvimpl;

extern "C" kv_status kv_store_fp8_ex(const void* k, const void* v, void* k_cache, void* v_cache,
                                     const void* indices, kv_index_dtype index_dtype,
                                     int64_t index_stride, int64_t num_tokens, int32_t num_heads,
                                     int32_t head_dim, kv_src_dtype src_dtype, const kv_strides* s,
                                     int64_t page_size, int64_t kc_page_stride,
                                     int64_t vc_page_stride, int64_t size_limit,
                                     kv_fp8_format format, kv_scale_mode scale_mode,
                                     const float* inv_k_scale, const float* inv_v_scale,
                                     float* k_scales, float* v_scales, int64_t scales_slot_stride,
                                     kv_error_record* d_err, kv_stream_t stream_) {
  if (format != KV_FP8_E4M3FN && format != KV_FP8_E5M2) return KV_ERR_INVALID_ARG;
  if (scale_mode != KV_SCALE_NONE && scale_mode != KV_SCALE_TENSOR && scale_mode != KV_SCALE_TOKEN &&
      scale_mode != KV_SCALE_TOKEN_HEAD && scale_mode != KV_SCALE_PAGE)
    return KV_ERR_INVALID_ARG;
  const int fmt = format == KV_FP8_E5M2 ? kFmtE5M2 : kFmtE4M3;
  if (scale_mode == KV_SCALE_PAGE && page_size < 1) return KV_ERR_INVALID_ARG;
  if (scale_mode == KV_SCALE_NONE || scale_mode == KV_SCALE_TENSOR || scale_mode == KV_SCALE_PAGE)
    return store_fp8_static(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_tokens,
                            num_heads, head_dim, src_dtype, s, page_size, kc_page_stride,
                            vc_page_stride, size_limit, inv_k_scale, inv_v_scale,
                            scale_mode == KV_SCALE_NONE ? 0 : 1,
                            scale_mode == KV_SCALE_PAGE ? page_size : 0, fmt, d_err, stream_);

  // dynamic scales
  if (num_tokens < 0) return KV_ERR_INVALID_ARG;
  if (num_tokens == 0) return KV_OK;
  if (!common_args_ok(k, v, k_cache, v_cache, indices, index_dtype, index_stride, num_heads,
                      head_dim, s, size_limit, d_err))
    return KV_ERR_INVALID_ARG;
  if (src_dtype != KV_SRC_F16 && src_dtype != KV_SRC_BF16) return KV_ERR_INVALID_ARG;
  if (page_size < 1) return KV_ERR_INVALID_ARG;
  const bool per_head = scale_mode == KV_SCALE_TOKEN_HEAD;
  if (!k_scales || !v_scales || ((u64(k_scales) | u64(v_scales)) & 3u) != 0) return KV_ERR_INVALID_ARG;
  if (scales_slot_stride < (per_head ? num_heads : 1)) return KV_ERR_INVALID_ARG;
  if ((u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token) | u64(s->k_head) | u64(s->v_head)) & 1u)
    return KV_ERR_INVALID_ARG;
  if (s->k_dim != 2 || s->v_dim != 2 || s->kc_dim != 1 || s->vc_dim != 1) return KV_ERR_UNSUPPORTED;
  if (num_tokens > (int64_t{1} << 40)) return KV_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  bool on_device = true;
  {
    const void* in[3] = {k, v, indices};
    const kv_status cs = classify_inputs(in, 3, &on_device);
    if (cs != KV_OK) return cs;
  }
  const bool flat = kc_page_stride == page_size * s->kc_slot && vc_page_stride == page_size * s->vc_slot;
  const bool bf16 = src_dtype == KV_SRC_BF16;

  // fast path: heads contiguous on both sides, 32-byte aligned input rows,
  // 16-byte aligned cache rows, rows of at most 128 chunks, and (per head) a
  // head of D/16 chunks with D/16 a power of two up to 32 and at most 16
  // heads (a paired warp holds 2 * H groups, one per lane)
  {
    const int64_t row = static_cast<int64_t>(num_heads) * head_dim;
    const bool contiguous = num_heads == 1 || (s->k_head == 2 * static_cast<int64_t>(head_dim) &&
                                               s->v_head == 2 * static_cast<int64_t>(head_dim) &&
                                               s->kc_head == head_dim && s->vc_head == head_dim);
    const uint64_t in_bits = u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token);
    uint64_t out_bits = u64(k_cache) | u64(v_cache) | u64(s->kc_slot) | u64(s->vc_slot);
    if (!flat) out_bits |= u64(kc_page_stride) | u64(vc_page_stride);
    const int64_t gch = head_dim / 16;
    const bool groups_ok = !per_head || (head_dim % 16 == 0 && gch <= 32 && (gch & (gch - 1)) == 0 &&
                                         2 * num_heads <= 32);
    const int64_t chunks = row / 16;
    // staged form: input rows of 512, 1024 or 2048 bytes in device memory,
    // 16-byte aligned; groups of a power-of-two number of pieces that split a
    // row into at most 16 groups
    const int64_t rb = 2 * row;  // input row bytes
    const int64_t gpieces = per_head ? head_dim / 8 : rb / 16;
    const bool staged_ok = KV_DYN_STAGED && on_device && contiguous &&
                           (rb == 512 || rb == 1024 || rb == 2048) &&
                           (in_bits & 15u) == 0 && (out_bits & 7u) == 0 &&
                           (!per_head || (head_dim % 8 == 0 && (gpieces & (gpieces - 1)) == 0 &&
                                          rb / 16 / gpieces <= 16));
    if (staged_ok) {
      StagedParams q = {};
      q.side[0] = DynSide{static_cast<const uint8_t*>(k), static_cast<uint8_t*>(k_cache),
                          s->k_token, s->k_head, s->kc_slot, s->kc_head,
                          flat ? s->kc_slot : kc_page_stride, k_scales};
      q.side[1] = DynSide{static_cast<const uint8_t*>(v), static_cast<uint8_t*>(v_cache),
                          s->v_token, s->v_head, s->vc_slot, s->vc_head,
                          flat ? s->vc_slot : vc_page_stride, v_scales};
      q.indices = indices;
      q.index_stride = index_stride;
      q.size_limit = size_limit;
      q.page_size = flat ? 1 : page_size;
      q.scales_stride = scales_slot_stride;
      q.num_tokens = num_tokens;
      q.row_bytes = static_cast<uint32_t>(rb);
      q.group_pieces = static_cast<uint32_t>(gpieces);
      int64_t stages = KV_DYN_STAGE_BYTES / (2 * rb);
      if (stages > static_cast<int64_t>(kDynMaxStages)) stages = kDynMaxStages;
      if (stages < 2) stages = 2;
      q.stages = static_cast<uint32_t>(stages);
      q.fmax = fmt == kFmtE5M2 ? 57344.0f : 448.0f;
      q.err = d_err;
      q.prefetch = 1;
      const int pieces = static_cast<int>(rb / 512);
      return index_dtype == KV_INDEX_I64 ? launch_dyn_staged<int64_t>(pieces, fmt, bf16, q, stream)
                                         : launch_dyn_staged<int32_t>(pieces, fmt, bf16, q, stream);
    }
    if (contiguous && row % 16 == 0 && chunks <= 128 && (in_bits & 31u) == 0 &&
        (out_bits & 15u) == 0 && groups_ok) {
      DynRowParams p = {};
      p.side[0] = DynSide{static_cast<const uint8_t*>(k), static_cast<uint8_t*>(k_cache),
                          s->k_token, s->k_head, s->kc_slot, s->kc_head,
                          flat ? s->kc_slot : kc_page_stride, k_scales};
      p.side[1] = DynSide{static_cast<const uint8_t*>(v), static_cast<uint8_t*>(v_cache),
                          s->v_token, s->v_head, s->vc_slot, s->vc_head,
                          flat ? s->vc_slot : vc_page_stride, v_scales};
      p.indices = indices;
      p.index_stride = index_stride;
      p.size_limit = size_limit;
      p.page_size = flat ? 1 : page_size;
      p.scales_stride = scales_slot_stride;
      p.shape.parts = 1;
      p.shape.units_per_side = 1;
      p.shape.units_per_token = 2;
      p.shape.num_units = static_cast<uint64_t>(num_tokens) * 2u;
      p.shape.part_chunks = static_cast<uint32_t>(chunks);
      p.chunks = static_cast<uint32_t>(chunks);
      p.group_chunks = per_head ? static_cast<uint32_t>(gch) : 0u;
      p.fmax = fmt == kFmtE5M2 ? 57344.0f : 448.0f;
      p.err = d_err;
      p.prefetch = on_device ? 1 : 0;
      const int j = chunks <= 32 ? 1 : chunks <= 64 ? 2 : 4;
      return index_dtype == KV_INDEX_I64 ? launch_dyn_row<int64_t>(j, fmt, bf16, p, stream)
                                         : launch_dyn_row<int32_t>(j, fmt, bf16, p, stream);
    }
  }

  // group layout: per head, or the whole row (one segment when heads are
  // contiguous on both sides, else one segment per head)
  const int64_t D = head_dim;
  const bool merged = !per_head && (num_heads == 1 || (s->k_head == 2 * D && s->v_head == 2 * D &&
                                                       s->kc_head == D && s->vc_head == D));
  const uint32_t groups = per_head ? static_cast<uint32_t>(num_heads) : 1u;
  const uint32_t gseg = (per_head || merged) ? 1u : static_cast<uint32_t>(num_heads);
  const int64_t seg_elems = merged ? D * num_heads : D;
  const bool segs_used = !merged;  // head strides address segments
  uint64_t sbits = u64(k) | u64(v) | u64(s->k_token) | u64(s->v_token);
  uint64_t dbits = u64(k_cache) | u64(v_cache) | u64(s->kc_slot) | u64(s->vc_slot);
  if (segs_used) {
    sbits |= u64(s->k_head) | u64(s->v_head);
    dbits |= u64(s->kc_head) | u64(s->vc_head);
  }
  if (!flat) dbits |= u64(kc_page_stride) | u64(vc_page_stride);
  // chunk of CH elements: 2*CH input bytes, CH output bytes; prefer enough
  // chunks per group to keep every lane busy
  int ch = 1;
  for (int c = 8; c >= 1; c >>= 1) {
    const bool ok = seg_elems % c == 0 && (sbits & static_cast<uint64_t>(2 * c - 1)) == 0 &&
                    (dbits & static_cast<uint64_t>(c - 1)) == 0;
    if (!ok) continue;
    ch = c;
    if (static_cast<int64_t>(gseg) * (seg_elems / c) >= 32) break;
  }

  DynParams p = {};
  p.side[0] = DynSide{static_cast<const uint8_t*>(k), static_cast<uint8_t*>(k_cache), s->k_token,
                      s->k_head, s->kc_slot, s->kc_head, flat ? s->kc_slot : kc_page_stride,
                      k_scales};
  p.side[1] = DynSide{static_cast<const uint8_t*>(v), static_cast<uint8_t*>(v_cache), s->v_token,
                      s->v_head, s->vc_slot, s->vc_head, flat ? s->vc_slot : vc_page_stride,
                      v_scales};
  p.indices = indices;
  p.index_stride = index_stride;
  p.size_limit = size_limit;
  p.page_size = flat ? 1 : page_size;
  p.scales_stride = scales_slot_stride;
  p.groups = groups;
  p.gseg = gseg;
  p.cps = static_cast<uint32_t>(seg_elems / ch);
  p.num_units = static_cast<uint64_t>(num_tokens) * 2u * groups;
  p.fmax = fmt == kFmtE5M2 ? 57344.0f : 448.0f;
  p.err = d_err;
  p.prefetch = (on_device && (sbits & 15u) == 0 && (seg_elems * 2) % 16 == 0) ? 1 : 0;
  return index_dtype == KV_INDEX_I64 ? launch_dyn<int64_t>(ch, fmt, bf16, p, stream)
                                     : launch_dyn<int32_t>(ch, fmt, bf16, p, stream);
}
