// Extended FP8 write: e4m3fn or e5m2 caches, and dynamic scales computed in
// the kernel per token row or per (token, head).
//
// The fused FP8 write's module docstring (sglang trtllm_fp8_kv_kernel.py)
// advertises scales computed per token or per page, but its kernel only
// takes a per-tensor scale; this file supplies the per-token form.  For each group
// (the K or V row of a token, or one head of it): amax = max |x| (NaN
// ignored); inv = fmax / amax and scale = amax / fmax in fp32 (both 1 when
// amax is 0); codes = fp8(x * inv); `scale` goes to the caller's per-slot
// scale cache.  fmax is 448 for e4m3fn and 57344 for e5m2.
//
// Two kernels.  kv_fp8_dyn_row takes rows whose heads are contiguous (the
// common layout): the static write's lane layout, each group's amax reduced
// over the lanes that hold it, one division per warp (see there).  The
// general kernel kv_fp8_dyn_rows takes every other layout: one warp owns one
// group, whose elements are loaded once into registers (up to 4 chunks per
// lane, 2 for 16-byte chunks; longer groups are re-read from L2 in a second
// pass); the warp reduces amax, then converts and stores the codes, and lane
// 0 stores the group's scale.  As in the other write kernels, the source
// bytes are prefetched into L2 before the programmatic-launch wait.
#include "kv_host.h"

#ifndef KV_DYN_LOOKAHEAD
#define KV_DYN_LOOKAHEAD 1   // multi-wave row launches: prefetch the unit one resident wave ahead
#endif

namespace kvimpl {
namespace {

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
#if KV_PACKED_MATH
    uint32_t pm = 0;
#pragma unroll
    for (int i = 0; i < CH / 2; ++i) pm = absmax_pair<kBF16>(pm, c.w[i]);
    m = fmaxf(m, absmax_pair_value<kBF16>(pm));
#else
#pragma unroll
    for (int i = 0; i < CH / 2; ++i) {
      const float2 x = widen2<kBF16>(c.w[i]);
      m = fmaxf(m, fmaxf(fabsf(x.x), fabsf(x.y)));
    }
#endif
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

// Maxima of |x| over the even and over the odd elements of a 32-byte chunk
// (16 elements), as the two 16-bit halves of one word: a tree of packed
// max.xorsign.abs steps.  The maximum of 16-bit inputs is one of them, so
// the values are exact; their sign bits are arbitrary (cleared by the
// reduction below).  A NaN element never wins over a number.
template <bool kBF16>
__device__ __forceinline__ uint32_t chunk_pairmax(const Chunk<32>& c) {
  const uint32_t a0 = absmax_pair<kBF16>(c.w[0], c.w[1]);
  const uint32_t a1 = absmax_pair<kBF16>(c.w[2], c.w[3]);
  const uint32_t a2 = absmax_pair<kBF16>(c.w[4], c.w[5]);
  const uint32_t a3 = absmax_pair<kBF16>(c.w[6], c.w[7]);
  return absmax_pair<kBF16>(absmax_pair<kBF16>(a0, a1), absmax_pair<kBF16>(a2, a3));
}

// Two pair maxima a, b folded into one word: max over a's halves in the low
// half, over b's in the high half.
template <bool kBF16>
__device__ __forceinline__ uint32_t fold_pairs(uint32_t a, uint32_t b) {
  return absmax_pair<kBF16>(__byte_perm(a, b, 0x5410), __byte_perm(a, b, 0x7632));
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
    amax = warp_absmax(amax);
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
// aligned run of D/16 lanes; xor shuffles over those lanes give its amax.  In
// the per-token mode the group is the whole row.  Large launches pair the K
// and the V row of a token in one warp (NS == 2).  The per-head and the
// per-token forms are separate instantiations (kHead), so each carries only
// its own reduction.
struct DynRowParams {
  DynSide side[2];
  const void* indices;
  int64_t index_stride, size_limit, page_size, scales_stride;
  UnitShape shape;          // units: (token, K|V) rows, or tokens when paired
  uint32_t chunks;          // 16-element chunks per row
  uint32_t group_chunks;    // chunks per scale group (D / 16, a power of two), or 0: the whole row
  float fmax;
  kv_error_record* err;
  int prefetch;             // rows in device memory: bulk L2 prefetch allowed
  uint64_t ahead;           // > 0: also prefetch the rows of unit u + ahead (set by launch_rows)
};

template <int J, int NS, bool kHead, typename IdxT, bool kBF16, int FMT>
__global__ void __launch_bounds__(kThreads, 65536 / (kThreads * (J * NS <= 4 ? 64 : 128)))
    kv_fp8_dyn_row(const __grid_constant__ DynRowParams p) {
  const uint32_t lane = threadIdx.x & 31u;
  const uint64_t nwarps = static_cast<uint64_t>(gridDim.x) * warps_per_cta();
  uint64_t u = static_cast<uint64_t>(blockIdx.x) * warps_per_cta() + (threadIdx.x >> 5);
  const uint32_t n = p.chunks;
  const uint32_t g = p.group_chunks;
  const uint32_t gsh = g != 0u ? static_cast<uint32_t>(__ffs(g) - 1) : 0u;  // log2(g)
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
    // the unit that takes this warp's place one resident wave later: its rows
    // go to L2 while this unit's reduction waits on its loads
    if (KV_DYN_LOOKAHEAD && kHead && p.ahead != 0 && lane == 0 && u + p.ahead < p.shape.num_units) {
      const Unit nx = decode_unit(p.shape, u + p.ahead);
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const DynSide& sd = p.side[NS == 2 ? i : nx.kv];
        prefetch_l2_bulk(sd.src + nx.token * sd.src_token, n * 32u);
      }
      prefetch_l2_line(static_cast<const IdxT*>(p.indices) + nx.token * p.index_stride);
    }
    // Group maxima.  Value t = i * J + j of a lane is side i's lane chunk j;
    // per head its group is the head of that chunk (g lanes hold it), per
    // token the side's row.  Each chunk's exact 16-bit maximum is packed two
    // to a word (value t in half t % 2 of word t / 2).
    //  - Per head, with at least 2V lanes to a group: a reduce-scatter over
    //    the group's lanes.  Each of the first log2(W) xor rounds hands the
    //    partner the half of the live words this lane does not keep, so one
    //    word (values 2b, 2b + 1) is left, and the remaining rounds reduce
    //    it over the lanes that kept the same word.
    //  - Per head with fewer lanes: every word is reduced over the group.
    //  - Per token: the sides' maxima in one word, reduced over the warp by
    //    redux.sync on fp32 copies (redux.sync over 8-lane masks measured
    //    slower than the shuffles; over the whole warp it is faster).
    constexpr int V = NS * J;
    constexpr int W = (V + 1) / 2;
    constexpr int S = W == 4 ? 2 : W == 2 ? 1 : 0;  // log2(W)
    const bool scatter = kHead && 2u * V <= g;
    float gm[V];       // per token: side t (t < NS); per head without scatter: the group of value t
    uint32_t word = 0u, wb = 0u;  // per head with scatter: the lane's word and its index
    {
      uint32_t b[V];
#pragma unroll
      for (int t = 0; t < V; ++t)
        b[t] = lane + 32u * (t % J) < n ? chunk_pairmax<kBF16>(buf[t / J][t % J]) : 0u;
      if constexpr (kHead) {
        uint32_t pk[W];
#pragma unroll
        for (int s = 0; s < W; ++s) pk[s] = 0u;
#pragma unroll
        for (int t = 0; t < V; ++t) {   // the chunk's maximum in both halves, kept in half t % 2
          const uint32_t m = absmax_pair<kBF16>(b[t], __byte_perm(b[t], 0u, 0x1032));
          pk[t / 2] |= m & ((t & 1) ? 0xFFFF0000u : 0x0000FFFFu);
        }
        if (scatter) {
#pragma unroll
          for (int k = 0; k < S; ++k) {
            const uint32_t o = g >> (k + 1);
            const bool up = (lane & o) != 0u;
#pragma unroll
            for (int x = 0; x < (W >> (k + 1)); ++x) {
              const uint32_t send = up ? pk[x] : pk[(W >> (k + 1)) + x];
              const uint32_t keep = up ? pk[(W >> (k + 1)) + x] : pk[x];
              pk[x] = absmax_pair<kBF16>(keep, __shfl_xor_sync(0xFFFFFFFFu, send, o));
            }
            if (up) wb += static_cast<uint32_t>(W >> (k + 1));
          }
          for (uint32_t o = g >> (S + 1); o > 0u; o >>= 1)
            pk[0] = absmax_pair<kBF16>(pk[0], __shfl_xor_sync(0xFFFFFFFFu, pk[0], o));
          word = pk[0];
        } else {
          for (uint32_t o = 1; o < g; o <<= 1)
#pragma unroll
            for (int s = 0; s < W; ++s) pk[s] = absmax_pair<kBF16>(pk[s], __shfl_xor_sync(0xFFFFFFFFu, pk[s], o));
#pragma unroll
          for (int s = 0; s < W; ++s) {
            const float2 x = widen2<kBF16>(pk[s]);
            gm[2 * s] = fabsf(x.x);
            if (2 * s + 1 < V) gm[2 * s + 1] = fabsf(x.y);
          }
        }
      } else {
        uint32_t side[NS];
#pragma unroll
        for (int i = 0; i < NS; ++i) {
          side[i] = b[i * J];
#pragma unroll
          for (int j = 1; j < J; ++j) side[i] = absmax_pair<kBF16>(side[i], b[i * J + j]);
        }
        const float2 x = widen2<kBF16>(fold_pairs<kBF16>(side[0], NS == 2 ? side[NS - 1] : 0u));
        gm[0] = warp_absmax(x.x);
        if (NS == 2) gm[NS - 1] = warp_absmax(x.y);
      }
    }
    if (slot < 0 || slot >= p.size_limit) {
      if (w.rank == 0 && lane == 0) record_oob(p.err, static_cast<uint64_t>(w.token));
      continue;
    }
    // Scales.  A group's two divisions (fmax / amax, its inverse scale, and
    // amax / fmax, its stored scale) go to two lanes that hold the group's
    // maximum, so the warp runs one division; every lane then takes its
    // chunks' inverse scales from the inverse-scale lanes.
    float inv[V];
    if constexpr (!kHead) {
      // lanes i and NS + i serve side i
      const float a = lane == 1u || lane == NS + 1u ? gm[NS - 1] : gm[0];
      const bool inv_role = lane < NS;
      const float res = a > 0.0f ? __fdiv_rn(inv_role ? p.fmax : a, inv_role ? a : p.fmax) : 1.0f;
      if (!inv_role && lane < 2u * NS) p.side[NS == 2 ? lane - NS : w.kv].scales[slot * p.scales_stride] = res;
#pragma unroll
      for (int t = 0; t < V; ++t) inv[t] = __shfl_sync(0xFFFFFFFFu, res, static_cast<uint32_t>(t / J));
    } else if (scatter) {
      // In the g lanes of a group block, lane r holds word wb: for V >= 2 it
      // serves value 2 wb + (r & 1), bit 1 of r picks the division; the lanes
      // with the same word and r below 4 (below 2 for V = 1) store scales.
      const uint32_t r = lane & (g - 1u);
      const uint32_t sub = r & ((g >> S) - 1u);
      const uint32_t t = V >= 2 ? 2u * wb + (r & 1u) : 0u;
      const bool scale_role = V >= 2 ? ((r >> 1) & 1u) != 0u : (r & 1u) != 0u;
      const float2 x = widen2<kBF16>(word);
      const float a = fabsf(V >= 2 && (r & 1u) ? x.y : x.x);
      const float res = a > 0.0f ? __fdiv_rn(scale_role ? a : p.fmax, scale_role ? p.fmax : a) : 1.0f;
      if (scale_role && sub < (V >= 2 ? 4u : 2u)) {
        const uint32_t j = t % J;
        const uint32_t first = 32u * j + (lane & ~(g - 1u));  // the group's first chunk
        if (first < n) p.side[NS == 2 ? t / J : w.kv].scales[slot * p.scales_stride + (first >> gsh)] = res;
      }
      const uint32_t base = lane & ~(g - 1u);
#pragma unroll
      for (int u2 = 0; u2 < V; ++u2) {
        // the inverse-scale lane of value u2: its word's scatter bits, and bit 0 = u2 & 1
        uint32_t rl = V >= 2 ? static_cast<uint32_t>(u2 & 1) : 0u;
#pragma unroll
        for (int k = 0; k < S; ++k)
          if ((u2 >> 1) & (W >> (k + 1))) rl += g >> (k + 1);
        inv[u2] = __shfl_sync(0xFFFFFFFFu, res, base + rl);
      }
    } else {
      // Small heads (fewer than 2V lanes to a group): the warp holds NS * gps
      // groups (gps per side); lane k forms both divisions of group k, its
      // maximum taken from the lane holding the group's first chunk, and
      // every lane takes its chunks' inverse scales from the owners.
      const uint32_t gps = n >> gsh;
      const uint32_t gk = lane % gps;          // lane's group within its side
      const uint32_t c0 = gk * g;              // first chunk of that group
      float amax_k = 0.0f;
#pragma unroll
      for (int t = 0; t < V; ++t) {
        const float v = __shfl_sync(0xFFFFFFFFu, gm[t], c0 % 32u);
        if (lane / gps == static_cast<uint32_t>(t / J) && c0 / 32u == static_cast<uint32_t>(t % J)) amax_k = v;
      }
      const bool pos_k = amax_k > 0.0f;
      const bool owner = lane < NS * gps;
      const float inv_k = owner && pos_k ? __fdiv_rn(p.fmax, amax_k) : 1.0f;
      if (owner) {
        const DynSide& sd = p.side[NS == 2 ? lane / gps : w.kv];
        sd.scales[slot * p.scales_stride + gk] = pos_k ? __fdiv_rn(amax_k, p.fmax) : 1.0f;
      }
#pragma unroll
      for (int t = 0; t < V; ++t) {
        const uint32_t k = static_cast<uint32_t>(t / J) * gps + ((lane + 32u * (t % J)) >> gsh);
        inv[t] = __shfl_sync(0xFFFFFFFFu, inv_k, k < 32u ? k : 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const DynSide& sd = p.side[NS == 2 ? i : w.kv];
      uint8_t* dst = sd.dst + paged_offset(slot, p.page_size, sd.dst_page, sd.dst_slot);
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const uint32_t c = lane + 32u * j;
        if (c < n) st_stream(dst + static_cast<size_t>(c) * 16u, chunk_quant<16, kBF16, FMT>(buf[i][j], inv[i * J + j]));
      }
    }
  }
  if (!KV_EARLY_TRIGGER) grid_dependents_launch();
}

// Per head, the warps of a multi-wave launch prefetch the rows one resident
// wave ahead (launch_rows sets params.ahead); per token the look-ahead
// measured slower and is compiled out.
template <int J, int NS, bool kHead, typename IdxT, int FMT>
kv_status launch_dyn_row_k(bool bf16, const DynRowParams& p, cudaStream_t stream, uint64_t bytes) {
  if constexpr (kHead) {
    if (bf16) return launch_rows(kv_fp8_dyn_row<J, NS, true, IdxT, true, FMT>, p.shape.num_units, p, stream, bytes);
    return launch_rows(kv_fp8_dyn_row<J, NS, true, IdxT, false, FMT>, p.shape.num_units, p, stream, bytes);
  } else {
    if (bf16) return launch(kv_fp8_dyn_row<J, NS, false, IdxT, true, FMT>, p.shape.num_units, p, stream);
    return launch(kv_fp8_dyn_row<J, NS, false, IdxT, false, FMT>, p.shape.num_units, p, stream);
  }
}

template <int J, typename IdxT, int FMT>
kv_status launch_dyn_row_j(bool bf16, const DynRowParams& p, cudaStream_t stream) {
  // bytes moved: each row's 32-byte input chunks read, 16-byte codes written
  const uint64_t bytes = p.shape.num_units * p.chunks * 48u;
  const bool head = p.group_chunks != 0;
  if (p.shape.num_units >= KV_LARGE_LAUNCH_WARPS) {
    DynRowParams q = p;   // one warp per token: K and V rows together
    q.shape.units_per_token = 1;
    q.shape.units_per_side = 1;
    q.shape.num_units /= 2;
    return head ? launch_dyn_row_k<J, 2, true, IdxT, FMT>(bf16, q, stream, bytes)
                : launch_dyn_row_k<J, 2, false, IdxT, FMT>(bf16, q, stream, bytes);
  }
  return head ? launch_dyn_row_k<J, 1, true, IdxT, FMT>(bf16, p, stream, bytes)
              : launch_dyn_row_k<J, 1, false, IdxT, FMT>(bf16, p, stream, bytes);
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
