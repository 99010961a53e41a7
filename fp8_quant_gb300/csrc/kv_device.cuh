// Device-side primitives shared by the KV-cache kernels (sm_103a): tuning
// constants, programmatic-launch hooks, L2 prefetch, streaming vector loads
// and stores, the unit decomposition and the FP8 conversion helpers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kv_abi.h"

// Tuning constants (defaults chosen by measurement on GB300).
#ifndef KV_THREADS
#define KV_THREADS 256          // threads per CTA of small (latency-bound) launches
#endif
#ifndef KV_THREADS_LARGE
#define KV_THREADS_LARGE 128    // threads per CTA of large launches
#endif
#ifndef KV_LARGE_LAUNCH_WARPS
#define KV_LARGE_LAUNCH_WARPS 4096  // a launch with at least this many warps of work is large
#endif
#ifndef KV_COPY_UNROLL
#define KV_COPY_UNROLL 4        // chunks per lane loaded before the first store
#endif
#ifndef KV_FP8_UNROLL
#define KV_FP8_UNROLL 2
#endif
#ifndef KV_FP8_MAX_OUT
#define KV_FP8_MAX_OUT 16       // widest FP8 output chunk per lane, bytes (16 or 32)
#endif
#ifndef KV_MAX_VEC
#define KV_MAX_VEC 32           // widest per-lane vector, bytes (32 = 256-bit ld/st)
#endif
#ifndef KV_EARLY_TRIGGER
#define KV_EARLY_TRIGGER 1      // let the next kernel on the stream launch at our start
#endif
#ifndef KV_L2_EVICT_FIRST
#define KV_L2_EVICT_FIRST 0     // evict-first L2 policy on the streamed loads and stores
#endif
#ifndef KV_GRID_WAVES
#define KV_GRID_WAVES 0         // grid cap in resident-capacity waves (0 = one warp per unit)
#endif
#ifndef KV_GATHER_PAIR
#define KV_GATHER_PAIR 1        // row gathers pair K and V per warp: 0 never, 1 large launches, 2 always
#endif
#ifndef KV_LOOKAHEAD
#define KV_LOOKAHEAD 1          // multi-wave gathers: each warp prefetches the unit one resident wave ahead
#endif
#ifndef KV_LOOKAHEAD_MAX_BYTES
#define KV_LOOKAHEAD_MAX_BYTES (64ull << 20)  // ... only when a launch moves at most this many bytes
#endif
#ifndef KV_PREFETCH
#define KV_PREFETCH 1           // L2 prefetch of the unit's source bytes before the grid wait
#endif
#ifndef KV_PACKED_MATH
#define KV_PACKED_MATH 1        // packed sm_100 arithmetic: f32x2 products, bf16x2/f16x2 maxima
#endif

namespace kvimpl {

constexpr int kThreads = KV_THREADS > KV_THREADS_LARGE ? KV_THREADS : KV_THREADS_LARGE;  // the most
constexpr int kMaxWarpsPerCta = kThreads / 32;
static_assert(KV_THREADS % 32 == 0 && KV_THREADS_LARGE % 32 == 0, "whole warps");
constexpr int kMaxDevices = 64;
static_assert(KV_MAX_VEC == 16 || KV_MAX_VEC == 32, "KV_MAX_VEC");

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Warps per CTA of the running launch (the host picks the CTA size per launch).
__device__ __forceinline__ uint32_t warps_per_cta() { return blockDim.x >> 5; }

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Every kernel's hand-over point: wait until the previous grid on the stream
// has completed and its memory is visible, and let the next kernel launch
// early.  The trigger only lets the next grid's CTAs become resident (and run
// their own pre-wait prologue); that grid still waits for this one to
// complete before it touches memory, so the trigger may come before the wait.
// The one-CTA bookkeeping kernels trigger first (kTriggerFirst): the big
// kernel after them then becomes resident, and prefetches, while the big
// kernel before them is still running (absmax 8.20 -> 7.87 us per call).
// The row kernels trigger after the wait: triggering first there let
// consecutive decode calls pile up waiting grids (1.50 -> 1.93 us per call).
template <bool kTriggerFirst = false>
__device__ __forceinline__ void grid_handover() {
  if (KV_EARLY_TRIGGER && kTriggerFirst) grid_dependents_launch();
  grid_dependency_wait();
  if (KV_EARLY_TRIGGER && !kTriggerFirst) grid_dependents_launch();
}

// L2 prefetch of `bytes` (a multiple of 16, 16-byte aligned) starting at p,
// issued by one thread.  Only warms L2, which is the point of coherence for
// every SM, so it may run before griddepcontrol.wait: a line the previous
// grid is still writing is updated in L2, and the real load comes after the
// wait.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Vector of VEC bytes moved by one lane.
template <int VEC> struct Chunk;
template <> struct Chunk<32> { uint32_t w[8]; };
template <> struct Chunk<16> { uint32_t w[4]; };
template <> struct Chunk<8> { uint32_t w[2]; };
template <> struct Chunk<4> { uint32_t w[1]; };
template <> struct Chunk<2> { uint16_t h; };
template <> struct Chunk<1> { uint16_t h; };

#if KV_L2_EVICT_FIRST
#define KV_L2_HINT ".L2::cache_hint"
#define KV_POLICY_ARG , "l"(l2_policy())
__device__ __forceinline__ uint64_t l2_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
#define KV_POL(n) ", %" #n
#else
#define KV_L2_HINT ""
#define KV_POLICY_ARG
#define KV_POL(n) ""
#endif

// Streaming loads: non-coherent path, no L1 allocation (each byte is read once).
__device__ __forceinline__ void ld_stream(Chunk<32>& c, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate" KV_L2_HINT
               ".v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8]" KV_POL(9) ";"
               : "=r"(c.w[0]), "=r"(c.w[1]), "=r"(c.w[2]), "=r"(c.w[3]), "=r"(c.w[4]),
                 "=r"(c.w[5]), "=r"(c.w[6]), "=r"(c.w[7])
               : "l"(p) KV_POLICY_ARG);
}
__device__ __forceinline__ void ld_stream(Chunk<16>& c, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate" KV_L2_HINT ".v4.u32 {%0, %1, %2, %3}, [%4]" KV_POL(5) ";"
               : "=r"(c.w[0]), "=r"(c.w[1]), "=r"(c.w[2]), "=r"(c.w[3])
               : "l"(p) KV_POLICY_ARG);
}
__device__ __forceinline__ void ld_stream(Chunk<8>& c, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(c.w[0]), "=r"(c.w[1])
               : "l"(p));
}
__device__ __forceinline__ void ld_stream(Chunk<4>& c, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(c.w[0]) : "l"(p));
}
__device__ __forceinline__ void ld_stream(Chunk<2>& c, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(c.h) : "l"(p));
}
__device__ __forceinline__ void ld_stream(Chunk<1>& c, const void* p) {
  asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(c.h) : "l"(p));
}

__device__ __forceinline__ void st_stream(void* p, const Chunk<32>& c) {
  asm volatile("st.global" KV_L2_HINT ".v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}" KV_POL(9) ";"
               ::"l"(p), "r"(c.w[0]), "r"(c.w[1]), "r"(c.w[2]), "r"(c.w[3]), "r"(c.w[4]),
               "r"(c.w[5]), "r"(c.w[6]), "r"(c.w[7]) KV_POLICY_ARG
               : "memory");
}
__device__ __forceinline__ void st_stream(void* p, const Chunk<16>& c) {
  asm volatile("st.global" KV_L2_HINT ".v4.u32 [%0], {%1, %2, %3, %4}" KV_POL(5) ";"
               ::"l"(p), "r"(c.w[0]), "r"(c.w[1]), "r"(c.w[2]), "r"(c.w[3]) KV_POLICY_ARG
               : "memory");
}
__device__ __forceinline__ void st_stream(void* p, const Chunk<8>& c) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(c.w[0]), "r"(c.w[1]) : "memory");
}
__device__ __forceinline__ void st_stream(void* p, const Chunk<4>& c) {
  asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(c.w[0]) : "memory");
}
__device__ __forceinline__ void st_stream(void* p, const Chunk<2>& c) {
  asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(c.h) : "memory");
}
__device__ __forceinline__ void st_stream(void* p, const Chunk<1>& c) {
  asm volatile("st.global.u8 [%0], %1;" ::"l"(p), "h"(c.h) : "memory");
}

template <typename IdxT>
__device__ __forceinline__ int64_t load_slot(const void* indices, int64_t stride, int64_t t) {
  return static_cast<int64_t>(__ldg(static_cast<const IdxT*>(indices) + t * stride));
}

// Slot id read before the programmatic-launch wait, at L2 only (no L1 line
// is filled, so the authoritative load after the wait cannot hit a stale
// copy).  The previous grid may still be writing it: the value is used only
// to aim an L2 prefetch, never to address a load or a store.
template <typename IdxT>
__device__ __forceinline__ int64_t speculative_slot(const void* indices, int64_t stride, int64_t t) {
  const IdxT* p = static_cast<const IdxT*>(indices) + t * stride;
  if constexpr (sizeof(IdxT) == 8) {
    long long v;
    asm volatile("ld.global.cg.s64 %0, [%1];" : "=l"(v) : "l"(p));
    return static_cast<int64_t>(v);
  } else {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return static_cast<int64_t>(v);
  }
}

// One record per skipped token: a count and the lowest skipped token (kept as
// its bitwise NOT so that a zeroed record means "none").
__device__ __forceinline__ void record_oob(kv_error_record* err, uint64_t t) {
  atomicAdd(reinterpret_cast<unsigned long long*>(&err->oob_count), 1ull);
  atomicMax(reinterpret_cast<unsigned long long*>(&err->first_bad_key),
            static_cast<unsigned long long>(~t));
}

// Unit u -> (token, K|V, segment, part).
struct UnitShape {
  uint64_t num_units;        // num_tokens * units_per_token
  uint32_t units_per_token;  // 2 * units_per_side
  uint32_t units_per_side;   // num_segments * parts
  uint32_t parts;            // parts per segment
  uint32_t part_chunks;      // chunks per part
};

struct Unit {
  int64_t token;
  uint32_t kv, seg, part, rank;  // rank: position of the unit inside its token
};

__device__ __forceinline__ Unit decode_unit(const UnitShape& s, uint64_t u) {
  Unit r;
  const uint64_t t = u / s.units_per_token;
  r.token = static_cast<int64_t>(t);
  r.rank = static_cast<uint32_t>(u - t * s.units_per_token);
  r.kv = r.rank >= s.units_per_side ? 1u : 0u;
  const uint32_t q = r.rank - r.kv * s.units_per_side;
  r.seg = q / s.parts;
  r.part = q - r.seg * s.parts;
  return r;
}

// Two fp32 values to two e4m3fn bytes (lo in bits 0-7): round to nearest even,
// saturate finite overflow and infinities to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Same for e5m2 (largest finite 57344; infinities saturate to it too).
__device__ __forceinline__ uint32_t e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// FP8 formats: the template parameter FMT of the conversion helpers.
constexpr int kFmtE4M3 = 0;
constexpr int kFmtE5M2 = 1;

template <int FMT>
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
  if constexpr (FMT == kFmtE5M2) return e5m2x2(lo, hi);
  return e4m3x2(lo, hi);
}

// Two packed 2-byte inputs -> fp32 (exact).
template <bool kBF16>
__device__ __forceinline__ float2 widen2(uint32_t w) {
  if constexpr (kBF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu))),
                       __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))));
  }
}

// x * s for both lanes of x: two IEEE fp32 products, round to nearest,
// subnormals kept -- with KV_PACKED_MATH one packed sm_100 instruction
// (mul.rn.f32x2) instead of two.
__device__ __forceinline__ float2 mul2_rn(float2 x, float s) {
#if KV_PACKED_MATH
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %4};\n\t"
      "mul.rn.f32x2 d, a, b;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(x.x), "f"(x.y), "f"(s));
  return r;
#else
  return make_float2(__fmul_rn(x.x, s), __fmul_rn(x.y, s));
#endif
}

template <bool kBF16, int FMT = kFmtE4M3>
__device__ __forceinline__ uint32_t quant2(uint32_t w, float inv) {
  const float2 y = mul2_rn(widen2<kBF16>(w), inv);
  return fp8x2<FMT>(y.x, y.y);
}

// Running maximum of |x| over packed pairs of 2-byte floats, lane by lane,
// in one instruction per pair: max.xorsign.abs keeps the larger magnitude
// (the sign bit is the XOR of the operands' signs, cleared when the value is
// read), and a NaN operand yields the other one, so NaN elements never win.
// Start from m = 0.
template <bool kBF16>
__device__ __forceinline__ uint32_t absmax_pair(uint32_t m, uint32_t w) {
  uint32_t r;
  if constexpr (kBF16) {
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w));
  } else {
    asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w));
  }
  return r;
}

// The larger magnitude of a running pair maximum, as fp32 (exact).
template <bool kBF16>
__device__ __forceinline__ float absmax_pair_value(uint32_t m) {
  const float2 x = widen2<kBF16>(m);
  return fmaxf(fabsf(x.x), fabsf(x.y));
}

// max |x| over the 32 lanes of a warp (all of them execute it): one
// redux.sync on fp32, which ignores NaN inputs (only NaN everywhere gives
// NaN).
__device__ __forceinline__ float warp_absmax(float x) {
  float r;
  asm volatile("redux.sync.max.abs.f32 %0, %1, %2;" : "=f"(r) : "f"(x), "r"(0xFFFFFFFFu));
  return r;
}

// One lane's chunk: OUT output bytes from OUT 2-byte inputs.
// Byte offset of cache row `slot`: (slot / page_size) * page_stride +
// (slot % page_size) * slot_stride.  page_size == 1 means a flat cache whose
// page stride is the slot stride.
__device__ __forceinline__ int64_t paged_offset(int64_t slot, int64_t page_size, int64_t page_stride,
                                                int64_t slot_stride) {
  if (page_size == 1) return slot * page_stride;
  const int64_t page = slot / page_size;
  return page * page_stride + (slot - page * page_size) * slot_stride;
}

}  // namespace kvimpl
