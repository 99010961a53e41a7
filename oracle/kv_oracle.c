/*
 * CPU oracle for the KV-cache write path -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct restatement of what the write path
 * computes, used to check the CUDA library.  Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant with the CUDA library, and the library never
 * calls it.
 *
 * Sources restated here (sglang):
 *   - kvcache.cuh, kernel `store_kvcache` and helper `copy_kv_warp`: each new
 *     token's K row and V row are copied byte for byte into the cache row
 *     named by `indices[token]`; the slot must satisfy 0 <= slot < size_limit.
 *   - trtllm_fp8_kv_kernel.py, kernels `_fused_fp8_set_kv_buffer_kernel` and
 *     `_process_kv_tensor`: slot -> (page_id = slot / page_size,
 *     page_offset = slot % page_size); each element is multiplied by the fp32
 *     inverse scale (when a scale is provided), converted to FP8 e4m3fn, and
 *     stored at page_id*stride_page + page_offset*stride_offset
 *     + head*stride_head + dim*stride_dim.
 *
 * Readings taken where the pages are silent (all stated again in the design
 * notes): out-of-range slots are skipped and counted instead of trapping; the
 * FP8 conversion rounds to nearest, ties to even, saturates to +-448 (+-Inf
 * included) and maps every NaN to 0x7F; a bf16/fp16 input widens exactly to
 * fp32 and the scale multiply is a single fp32 rounding.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define KVO_OK 0
#define KVO_ERR_ARG 1

/* ------------------------------------------------------------------------ */
/* Number formats.                                                          */
/* ------------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32: widening is exact. */
float kvo_bf16_to_f32(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/* IEEE binary16: 1 sign, 5 exponent bits (bias 15), 10 fraction bits.
 * Value = (-1)^s * 2^(e-15) * (1 + f/1024) for 1 <= e <= 30,
 *         (-1)^s * 2^-14 * (f/1024) for e == 0, Inf/NaN for e == 31. */
float kvo_f16_to_f32(uint16_t bits)
{
    int s = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1F;
    int f = bits & 0x3FF;
    double mag;
    if (e == 0x1F) {
        mag = f ? NAN : INFINITY;
    } else if (e == 0) {
        mag = ldexp((double)f, -24);
    } else {
        mag = ldexp(1024.0 + (double)f, e - 25);
    }
    return (float)(s ? -mag : mag);
}

/* FP8 e4m3fn (OCP 8-bit floating point, E4M3): 1 sign, 4 exponent bits
 * (bias 7), 3 mantissa bits; no infinities; S.1111.111 is NaN, so the
 * largest finite magnitude is S.1111.110 = 1.75 * 2^8 = 448.
 * Value = (-1)^s * 2^(E-7) * (1 + m/8) for E >= 1, (-1)^s * 2^-6 * (m/8)
 * for E == 0.  Returns the exact value (NaN for the two NaN codes). */
double kvo_e4m3fn_decode(uint8_t code)
{
    int s = code >> 7;
    int E = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (E == 0xF && m == 0x7)
        return NAN;
    if (E == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(8.0 + (double)m, E - 10);
    return s ? -mag : mag;
}

#define KVO_E4M3_NAN 0x7F       /* every NaN input maps to this code */
#define KVO_E4M3_MAXFIN 0x7E    /* 448 */

/* Round y to the nearest e4m3fn value, ties to the even mantissa, saturating
 * finite overflow and infinities to +-448.  Works in float64, where every
 * fp32 input and every e4m3fn value is exact, so the only rounding is the
 * explicit nearest-even step below. */
uint8_t kvo_e4m3fn_encode(float y)
{
    double a = fabs((double)y);
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    if (isnan(y))
        return KVO_E4M3_NAN;
    if (a >= 448.0)
        return sign | KVO_E4M3_MAXFIN;
    if (a < 0x1p-6) {
        /* Subnormal range: multiples of 2^-9.  q = a / 2^-9 is exact. */
        double q = a * 0x1p9;
        double m = nearbyint(q);       /* default mode: nearest, ties even */
        /* m == 8 is the smallest normal, 2^-6, whose code is also 8. */
        return sign | (uint8_t)m;
    }
    int ex;
    (void)frexp(a, &ex);               /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                    /* a in [2^e, 2^(e+1)), e in [-6, 8] */
    double q = ldexp(a, 3 - e);        /* in [8, 16), exact */
    double m = nearbyint(q);           /* in [8, 16] */
    if (m == 16.0) {                   /* mantissa carry into the exponent */
        m = 8.0;
        e += 1;
    }
    int code = ((e + 7) << 3) | ((int)m - 8);
    if (code > KVO_E4M3_MAXFIN)        /* cannot happen for a < 448 */
        code = KVO_E4M3_MAXFIN;
    return sign | (uint8_t)code;
}

/* Round a float to bf16 (IEEE binary32's sign and 8 exponent bits, 7 stored
 * fraction bits): nearest, ties to even; overflow rounds to +-Inf; every NaN
 * becomes the canonical 0x7FFF.  Same plain method as the e4m3fn encoder:
 * scale the magnitude so the kept bits are the integer part, round once. */
uint16_t kvo_f32_to_bf16(float x)
{
    double a = fabs((double)x);
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    if (isnan(x))
        return 0x7FFF;
    if (isinf(x))
        return sign | 0x7F80;
    if (a < 0x1p-126) {                /* subnormal: multiples of 2^-133 */
        double m = nearbyint(a * 0x1p133);
        return sign | (uint16_t)m;     /* m == 128 is the smallest normal */
    }
    int ex;
    (void)frexp(a, &ex);
    int e = ex - 1;                    /* a in [2^e, 2^(e+1)) */
    double m = nearbyint(ldexp(a, 7 - e));   /* in [128, 256] */
    if (m == 256.0) {
        m = 128.0;
        e += 1;
    }
    if (e > 127)
        return sign | 0x7F80;
    return sign | (uint16_t)(((e + 127) << 7) | ((int)m - 128));
}

/* Round a float to IEEE binary16 (5 exponent bits, bias 15, 10 fraction
 * bits): nearest, ties to even; overflow rounds to +-Inf; every NaN becomes
 * the canonical 0x7FFF. */
uint16_t kvo_f32_to_f16(float x)
{
    double a = fabs((double)x);
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    if (isnan(x))
        return 0x7FFF;
    if (isinf(x))
        return sign | 0x7C00;
    if (a < 0x1p-14) {                 /* subnormal: multiples of 2^-24 */
        double m = nearbyint(a * 0x1p24);
        return sign | (uint16_t)m;     /* m == 1024 is the smallest normal */
    }
    int ex;
    (void)frexp(a, &ex);
    int e = ex - 1;
    double m = nearbyint(ldexp(a, 10 - e));  /* in [1024, 2048] */
    if (m == 2048.0) {
        m = 1024.0;
        e += 1;
    }
    if (e > 15)
        return sign | 0x7C00;
    return sign | (uint16_t)(((e + 15) << 10) | ((int)m - 1024));
}

/* fp32 product of the widened input and the fp32 inverse scale: the exact
 * float64 product of two floats rounded once to float. */
float kvo_scale_f32(float x, float inv)
{
    return (float)((double)x * (double)inv);
}

/* ------------------------------------------------------------------------ */
/* Index read and bounds rule.                                              */
/* ------------------------------------------------------------------------ */

static int64_t read_index(const void *indices, int index_is_i64, int64_t index_stride, int64_t t)
{
    if (index_is_i64)
        return ((const int64_t *)indices)[t * index_stride];
    return (int64_t)((const int32_t *)indices)[t * index_stride];
}

static void note_bad(int64_t t, int64_t *bad_count, int64_t *first_bad)
{
    if (*bad_count == 0 || t < *first_bad)
        *first_bad = t;
    *bad_count += 1;
}

/* ------------------------------------------------------------------------ */
/* Plain copy: kvcache.cuh `store_kvcache`.                                 */
/* strides[12], all in bytes:                                               */
/*   k_token, k_head, k_dim, v_token, v_head, v_dim,                        */
/*   kc_slot, kc_head, kc_dim, vc_slot, vc_head, vc_dim.                    */
/* Tokens [t_begin, t_end) are processed.  Returns KVO_OK or KVO_ERR_ARG;   */
/* *bad_count / *first_bad report tokens whose slot is out of range.        */
/* ------------------------------------------------------------------------ */
int kvo_store_copy(const uint8_t *k, const uint8_t *v, uint8_t *k_cache, uint8_t *v_cache,
                   const void *indices, int index_is_i64, int64_t index_stride,
                   int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                   int32_t elem_bytes, const int64_t *strides, int64_t size_limit,
                   int64_t *bad_count, int64_t *first_bad)
{
    if (elem_bytes <= 0 || num_heads <= 0 || head_dim <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v : k;
            uint8_t *dst = kv ? v_cache : k_cache;
            const int64_t *ss = strides + 3 * kv;       /* token, head, dim */
            const int64_t *ds = strides + 6 + 3 * kv;   /* slot, head, dim */
            for (int32_t h = 0; h < num_heads; ++h)
                for (int32_t d = 0; d < head_dim; ++d)
                    memcpy(dst + slot * ds[0] + h * ds[1] + d * ds[2],
                           src + t * ss[0] + h * ss[1] + d * ss[2], (size_t)elem_bytes);
        }
    }
    return KVO_OK;
}

/* Paged plain copy: trtllm_fp8_kv_kernel.py `_naive_fp8_set_kv_buffer` with a
 * 4-D cache [pages, page_size, H, D] of the input's dtype, where the write is
 * k_cache[slot // page_size, slot % page_size] = k[t].  Slot s lands at
 * (s / page_size) * page_stride + (s % page_size) * slot_stride. */
int kvo_store_copy_paged(const uint8_t *k, const uint8_t *v, uint8_t *k_cache, uint8_t *v_cache,
                         const void *indices, int index_is_i64, int64_t index_stride,
                         int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                         int32_t elem_bytes, const int64_t *strides, int64_t page_size,
                         int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                         int64_t *bad_count, int64_t *first_bad)
{
    if (elem_bytes <= 0 || num_heads <= 0 || head_dim <= 0 || page_size <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        int64_t page_id = slot / page_size;
        int64_t page_offset = slot % page_size;
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v : k;
            uint8_t *dst = kv ? v_cache : k_cache;
            const int64_t *ss = strides + 3 * kv;
            const int64_t *ds = strides + 6 + 3 * kv;
            int64_t page_stride = kv ? vc_page_stride : kc_page_stride;
            for (int32_t h = 0; h < num_heads; ++h)
                for (int32_t d = 0; d < head_dim; ++d)
                    memcpy(dst + page_id * page_stride + page_offset * ds[0] + h * ds[1] + d * ds[2],
                           src + t * ss[0] + h * ss[1] + d * ss[2], (size_t)elem_bytes);
        }
    }
    return KVO_OK;
}

/* ------------------------------------------------------------------------ */
/* Fused FP8 write: trtllm_fp8_kv_kernel.py `_fused_fp8_set_kv_buffer_kernel`
 * and `_process_kv_tensor`.  Inputs are bf16 (src_is_bf16 = 1) or fp16.
 * The cache element is one e4m3fn byte; strides as for kvo_store_copy, plus
 * the page strides of the two caches.  With use_scale == 0 the value is
 * converted unscaled. */
/* ------------------------------------------------------------------------ */
int kvo_store_fp8(const uint8_t *k, const uint8_t *v, uint8_t *k_cache, uint8_t *v_cache,
                  const void *indices, int index_is_i64, int64_t index_stride,
                  int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                  int src_is_bf16, const int64_t *strides, int64_t page_size,
                  int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                  float inv_k, float inv_v, int use_scale,
                  int64_t *bad_count, int64_t *first_bad)
{
    if (num_heads <= 0 || head_dim <= 0 || page_size <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        int64_t page_id = slot / page_size;
        int64_t page_offset = slot % page_size;
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v : k;
            uint8_t *dst = kv ? v_cache : k_cache;
            const int64_t *ss = strides + 3 * kv;
            const int64_t *ds = strides + 6 + 3 * kv;
            int64_t page_stride = kv ? vc_page_stride : kc_page_stride;
            float inv = kv ? inv_v : inv_k;
            for (int32_t h = 0; h < num_heads; ++h) {
                for (int32_t d = 0; d < head_dim; ++d) {
                    uint16_t bits;
                    memcpy(&bits, src + t * ss[0] + h * ss[1] + d * ss[2], sizeof bits);
                    float x = src_is_bf16 ? kvo_bf16_to_f32(bits) : kvo_f16_to_f32(bits);
                    float y = use_scale ? kvo_scale_f32(x, inv) : x;
                    dst[page_id * page_stride + page_offset * ds[0] + h * ds[1] + d * ds[2]] =
                        kvo_e4m3fn_encode(y);
                }
            }
        }
    }
    return KVO_OK;
}

/* Element-wise conversion helpers for the tests: n values in, n codes out. */
void kvo_encode_f32_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_e4m3fn_encode(x[i]);
}

void kvo_decode_array(const uint8_t *codes, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_e4m3fn_decode(codes[i]);
}

/* ------------------------------------------------------------------------ */
/* Inverse path: gather cache rows back into token-major rows.              */
/* The local counterpart of the gather-materialise step of                  */
/* dcp_direct_kv_gather.cu (`materialize_kv_gather_kernel`): row t of the   */
/* output takes the cache row named by indices[t].  strides: k_* / v_*      */
/* describe the OUTPUT rows, kc_* / vc_* the caches.  Out-of-range slots    */
/* leave the output row untouched and are counted.                          */
/* ------------------------------------------------------------------------ */
int kvo_gather_copy(const uint8_t *k_cache, const uint8_t *v_cache, uint8_t *k_out, uint8_t *v_out,
                    const void *indices, int index_is_i64, int64_t index_stride,
                    int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                    int32_t elem_bytes, const int64_t *strides, int64_t size_limit,
                    int64_t *bad_count, int64_t *first_bad)
{
    if (elem_bytes <= 0 || num_heads <= 0 || head_dim <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v_cache : k_cache;
            uint8_t *dst = kv ? v_out : k_out;
            const int64_t *os = strides + 3 * kv;
            const int64_t *cs = strides + 6 + 3 * kv;
            for (int32_t h = 0; h < num_heads; ++h)
                for (int32_t d = 0; d < head_dim; ++d)
                    memcpy(dst + t * os[0] + h * os[1] + d * os[2],
                           src + slot * cs[0] + h * cs[1] + d * cs[2], (size_t)elem_bytes);
        }
    }
    return KVO_OK;
}

/* Paged gather (the inverse of the paged copy): slot s is read at
 * (s / page_size) * page_stride + (s % page_size) * slot_stride + ... . */
int kvo_gather_copy_paged(const uint8_t *k_cache, const uint8_t *v_cache, uint8_t *k_out,
                          uint8_t *v_out, const void *indices, int index_is_i64,
                          int64_t index_stride, int64_t t_begin, int64_t t_end, int32_t num_heads,
                          int32_t head_dim, int32_t elem_bytes, const int64_t *strides,
                          int64_t page_size, int64_t kc_page_stride, int64_t vc_page_stride,
                          int64_t size_limit, int64_t *bad_count, int64_t *first_bad)
{
    if (elem_bytes <= 0 || num_heads <= 0 || head_dim <= 0 || page_size <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        int64_t page_id = slot / page_size;
        int64_t page_offset = slot % page_size;
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v_cache : k_cache;
            uint8_t *dst = kv ? v_out : k_out;
            const int64_t *os = strides + 3 * kv;
            const int64_t *cs = strides + 6 + 3 * kv;
            int64_t page_stride = kv ? vc_page_stride : kc_page_stride;
            for (int32_t h = 0; h < num_heads; ++h)
                for (int32_t d = 0; d < head_dim; ++d)
                    memcpy(dst + t * os[0] + h * os[1] + d * os[2],
                           src + page_id * page_stride + page_offset * cs[0] + h * cs[1] + d * cs[2],
                           (size_t)elem_bytes);
        }
    }
    return KVO_OK;
}

/* FP8 gather with dequantisation: each e4m3fn code is decoded exactly,
 * multiplied by the fp32 scale (when use_scale), and rounded to bf16
 * (out_is_bf16) or fp16.  The cache address of slot s is
 * (s / page_size) * page_stride + (s % page_size) * slot_stride + ...,
 * as in the forward write. */
int kvo_gather_fp8(const uint8_t *k_cache, const uint8_t *v_cache, uint8_t *k_out, uint8_t *v_out,
                   const void *indices, int index_is_i64, int64_t index_stride,
                   int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                   int out_is_bf16, const int64_t *strides, int64_t page_size,
                   int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                   float scale_k, float scale_v, int use_scale,
                   int64_t *bad_count, int64_t *first_bad)
{
    if (num_heads <= 0 || head_dim <= 0 || page_size <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        int64_t page_id = slot / page_size;
        int64_t page_offset = slot % page_size;
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v_cache : k_cache;
            uint8_t *dst = kv ? v_out : k_out;
            const int64_t *os = strides + 3 * kv;
            const int64_t *cs = strides + 6 + 3 * kv;
            int64_t page_stride = kv ? vc_page_stride : kc_page_stride;
            float scale = kv ? scale_v : scale_k;
            for (int32_t h = 0; h < num_heads; ++h) {
                for (int32_t d = 0; d < head_dim; ++d) {
                    uint8_t q = src[page_id * page_stride + page_offset * cs[0] + h * cs[1] + d * cs[2]];
                    float x = (float)kvo_e4m3fn_decode(q);
                    float y = use_scale ? kvo_scale_f32(x, scale) : x;
                    uint16_t bits = out_is_bf16 ? kvo_f32_to_bf16(y) : kvo_f32_to_f16(y);
                    memcpy(dst + t * os[0] + h * os[1] + d * os[2], &bits, sizeof bits);
                }
            }
        }
    }
    return KVO_OK;
}

void kvo_f32_to_bf16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_f32_to_bf16(x[i]);
}

void kvo_f32_to_f16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_f32_to_f16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Scale preparation.                                                       */
/* ------------------------------------------------------------------------ */

/* trtllm_fp8_kv_kernel.py, `fused_fp8_set_kv_buffer`: the inverse scale
 * 1.0 / scale is formed on the device in fp32 (so that no host sync is needed
 * during graph capture).  The float64 quotient of two floats rounded once to
 * float is the correctly rounded fp32 quotient. */
float kvo_inv_scale(float scale)
{
    return (float)(1.0 / (double)scale);
}

/* Per-tensor absolute maximum of the K rows and of the V rows (NaN elements
 * are ignored; an all-NaN or empty tensor gives 0) and the inverse scale
 * fp8_max / amax in fp32 (1.0 when amax is 0): the recipe of the fp8
 * workload's per-tensor scale, inv = 448 / amax for e4m3fn.
 * strides: the first six entries of the usual twelve (K and V rows). */
void kvo_absmax_inv(const uint8_t *k, const uint8_t *v, int src_is_bf16, int64_t num_tokens,
                    int32_t num_heads, int32_t head_dim, const int64_t *strides, float fp8_max,
                    float *amax_out, float *inv_out)
{
    for (int kv = 0; kv < 2; ++kv) {
        const uint8_t *src = kv ? v : k;
        const int64_t *ss = strides + 3 * kv;
        double amax = 0.0;
        for (int64_t t = 0; t < num_tokens; ++t)
            for (int32_t h = 0; h < num_heads; ++h)
                for (int32_t d = 0; d < head_dim; ++d) {
                    uint16_t bits;
                    memcpy(&bits, src + t * ss[0] + h * ss[1] + d * ss[2], sizeof bits);
                    double x = src_is_bf16 ? kvo_bf16_to_f32(bits) : kvo_f16_to_f32(bits);
                    if (!isnan(x) && fabs(x) > amax)
                        amax = fabs(x);
                }
        amax_out[kv] = (float)amax;
        inv_out[kv] = amax > 0.0 ? (float)((double)fp8_max / amax) : 1.0f;
    }
}

/* ------------------------------------------------------------------------ */
/* FP8 e5m2, and the extended FP8 write with dynamic per-group scales.      */
/* ------------------------------------------------------------------------ */

/* FP8 E5M2 (OCP 8-bit floating point): 1 sign, 5 exponent bits (bias 15), 2
 * mantissa bits; E = 31 holds +-Inf (m = 0) and NaN (m != 0); largest finite
 * magnitude 1.75 * 2^15 = 57344.  Value = 2^(E-15) * (1 + m/4) for
 * 1 <= E <= 30, 2^-14 * (m/4) for E = 0. */
double kvo_e5m2_decode(uint8_t code)
{
    int s = code >> 7;
    int E = (code >> 2) & 0x1F;
    int m = code & 0x3;
    double mag;
    if (E == 0x1F)
        return m ? NAN : (s ? -INFINITY : INFINITY);
    if (E == 0)
        mag = ldexp((double)m, -16);
    else
        mag = ldexp(4.0 + (double)m, E - 17);
    return s ? -mag : mag;
}

#define KVO_E5M2_NAN 0x7F
#define KVO_E5M2_MAXFIN 0x7B   /* 57344 */

/* Nearest e5m2 value, ties to even mantissa, finite overflow and +-Inf
 * saturated to +-57344 (the same satfinite rule as the e4m3fn encoder), every
 * NaN to 0x7F. */
uint8_t kvo_e5m2_encode(float y)
{
    double a = fabs((double)y);
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    if (isnan(y))
        return KVO_E5M2_NAN;
    if (a >= 57344.0)
        return sign | KVO_E5M2_MAXFIN;
    if (a < 0x1p-14) {                 /* subnormal: multiples of 2^-16 */
        double m = nearbyint(a * 0x1p16);
        return sign | (uint8_t)m;      /* m == 4 is the smallest normal */
    }
    int ex;
    (void)frexp(a, &ex);
    int e = ex - 1;
    double m = nearbyint(ldexp(a, 2 - e));   /* in [4, 8] */
    if (m == 8.0) {
        m = 4.0;
        e += 1;
    }
    int code = ((e + 15) << 2) | ((int)m - 4);
    if (code > KVO_E5M2_MAXFIN)
        code = KVO_E5M2_MAXFIN;
    return sign | (uint8_t)code;
}

void kvo_e5m2_encode_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_e5m2_encode(x[i]);
}

void kvo_e5m2_decode_array(const uint8_t *codes, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_e5m2_decode(codes[i]);
}

/* Extended FP8 write.  fmt: 0 e4m3fn, 1 e5m2.  scale_mode: 0 none, 1 one fp32
 * inverse scale per tensor (inv_k / inv_v), 2 dynamic per token row, 3
 * dynamic per (token, head), 4 one fp32 inverse scale per cache page, read
 * from k_scales[page_id] / v_scales[page_id] (page_id = slot / page_size, the
 * page of the fused FP8 write's `_process_kv_tensor`): the codes are
 * enc(fl32(x * inv[page_id])).  Dynamic: over the group's elements x (the whole
 * K row of the token, or one head of it), amax = max |x| (NaN ignored); when
 * amax > 0, inv = fl32(fmax / amax) and scale = fl32(amax / fmax), else both
 * are 1; the codes are enc(fl32(x * inv)) and `scale` is stored at
 * k_scales[slot * scales_slot_stride + g] (g = head for mode 3, 0 for mode 2),
 * likewise for V.  fmax is 448 (e4m3fn) or 57344 (e5m2).  This is the
 * "per-token scale computation" the fused FP8 write's module docstring
 * (trtllm_fp8_kv_kernel.py) names and does not implement; the reading above is
 * this library's. */
int kvo_store_fp8_ex(const uint8_t *k, const uint8_t *v, uint8_t *k_cache, uint8_t *v_cache,
                     const void *indices, int index_is_i64, int64_t index_stride,
                     int64_t t_begin, int64_t t_end, int32_t num_heads, int32_t head_dim,
                     int src_is_bf16, const int64_t *strides, int64_t page_size,
                     int64_t kc_page_stride, int64_t vc_page_stride, int64_t size_limit,
                     int fmt, int scale_mode, float inv_k, float inv_v, float *k_scales,
                     float *v_scales, int64_t scales_slot_stride,
                     int64_t *bad_count, int64_t *first_bad)
{
    if (num_heads <= 0 || head_dim <= 0 || page_size <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    if (fmt < 0 || fmt > 1 || scale_mode < 0 || scale_mode > 4)
        return KVO_ERR_ARG;
    const double fmax = fmt ? 57344.0 : 448.0;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        int64_t page_id = slot / page_size;
        int64_t page_offset = slot % page_size;
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v : k;
            uint8_t *dst = kv ? v_cache : k_cache;
            const int64_t *ss = strides + 3 * kv;
            const int64_t *ds = strides + 6 + 3 * kv;
            int64_t page_stride = kv ? vc_page_stride : kc_page_stride;
            float *scales = kv ? v_scales : k_scales;
            int groups = scale_mode == 3 ? num_heads : 1;
            int heads_per_group = scale_mode == 3 ? 1 : num_heads;
            for (int g = 0; g < groups; ++g) {
                float inv = 1.0f;
                if (scale_mode == 1) {
                    inv = kv ? inv_v : inv_k;
                } else if (scale_mode == 4) {
                    inv = scales[page_id];
                } else if (scale_mode >= 2) {
                    double amax = 0.0;
                    for (int32_t hh = 0; hh < heads_per_group; ++hh)
                        for (int32_t d = 0; d < head_dim; ++d) {
                            int32_t h = g * heads_per_group + hh;
                            uint16_t bits;
                            memcpy(&bits, src + t * ss[0] + h * ss[1] + d * ss[2], sizeof bits);
                            double x = src_is_bf16 ? kvo_bf16_to_f32(bits) : kvo_f16_to_f32(bits);
                            if (!isnan(x) && fabs(x) > amax)
                                amax = fabs(x);
                        }
                    float scale = 1.0f;
                    if (amax > 0.0) {
                        inv = (float)(fmax / amax);     /* correctly rounded fp32 quotients */
                        scale = (float)(amax / fmax);
                    }
                    scales[slot * scales_slot_stride + g] = scale;
                }
                for (int32_t hh = 0; hh < heads_per_group; ++hh)
                    for (int32_t d = 0; d < head_dim; ++d) {
                        int32_t h = g * heads_per_group + hh;
                        uint16_t bits;
                        memcpy(&bits, src + t * ss[0] + h * ss[1] + d * ss[2], sizeof bits);
                        float x = src_is_bf16 ? kvo_bf16_to_f32(bits) : kvo_f16_to_f32(bits);
                        float y = scale_mode ? kvo_scale_f32(x, inv) : x;
                        dst[page_id * page_stride + page_offset * ds[0] + h * ds[1] + d * ds[2]] =
                            fmt ? kvo_e5m2_encode(y) : kvo_e4m3fn_encode(y);
                    }
            }
        }
    }
    return KVO_OK;
}

/* Extended dequantising gather: codes of format fmt decoded exactly, times
 * the scale (mode 0: none; 1: scale_k / scale_v per tensor; 2/3: the per-slot
 * scale k_scales[slot * scales_slot_stride + g] written by the extended
 * write; 4: the per-page scale k_scales[slot / page_size]), rounded to
 * bf16 / fp16. */
int kvo_gather_fp8_ex(const uint8_t *k_cache, const uint8_t *v_cache, uint8_t *k_out,
                      uint8_t *v_out, const void *indices, int index_is_i64,
                      int64_t index_stride, int64_t t_begin, int64_t t_end, int32_t num_heads,
                      int32_t head_dim, int out_is_bf16, const int64_t *strides,
                      int64_t page_size, int64_t kc_page_stride, int64_t vc_page_stride,
                      int64_t size_limit, int fmt, int scale_mode, float scale_k,
                      float scale_v, const float *k_scales, const float *v_scales,
                      int64_t scales_slot_stride, int64_t *bad_count, int64_t *first_bad)
{
    if (num_heads <= 0 || head_dim <= 0 || page_size <= 0 || t_begin > t_end)
        return KVO_ERR_ARG;
    if (fmt < 0 || fmt > 1 || scale_mode < 0 || scale_mode > 4)
        return KVO_ERR_ARG;
    *bad_count = 0;
    *first_bad = -1;
    for (int64_t t = t_begin; t < t_end; ++t) {
        int64_t slot = read_index(indices, index_is_i64, index_stride, t);
        if (slot < 0 || slot >= size_limit) {
            note_bad(t, bad_count, first_bad);
            continue;
        }
        int64_t page_id = slot / page_size;
        int64_t page_offset = slot % page_size;
        for (int kv = 0; kv < 2; ++kv) {
            const uint8_t *src = kv ? v_cache : k_cache;
            uint8_t *dst = kv ? v_out : k_out;
            const int64_t *os = strides + 3 * kv;
            const int64_t *cs = strides + 6 + 3 * kv;
            int64_t page_stride = kv ? vc_page_stride : kc_page_stride;
            const float *scales = kv ? v_scales : k_scales;
            for (int32_t h = 0; h < num_heads; ++h) {
                float scale = 1.0f;
                if (scale_mode == 1)
                    scale = kv ? scale_v : scale_k;
                else if (scale_mode == 4)
                    scale = scales[page_id];
                else if (scale_mode >= 2)
                    scale = scales[slot * scales_slot_stride + (scale_mode == 3 ? h : 0)];
                for (int32_t d = 0; d < head_dim; ++d) {
                    uint8_t q = src[page_id * page_stride + page_offset * cs[0] + h * cs[1] + d * cs[2]];
                    float x = (float)(fmt ? kvo_e5m2_decode(q) : kvo_e4m3fn_decode(q));
                    float y = scale_mode ? kvo_scale_f32(x, scale) : x;
                    uint16_t bits = out_is_bf16 ? kvo_f32_to_bf16(y) : kvo_f32_to_f16(y);
                    memcpy(dst + t * os[0] + h * os[1] + d * os[2], &bits, sizeof bits);
                }
            }
        }
    }
    return KVO_OK;
}
