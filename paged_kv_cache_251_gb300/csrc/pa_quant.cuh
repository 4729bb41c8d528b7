// 8-bit KV cache: the row quantiser and exact code -> fp32 widening.
//
// Sources: "KV Cache与长上下文管理", KV-cache quantisation (FP16 -> INT8 -> INT4:
// the cache stored in 8 bits halves its size) and the mjmagnets article,
// section 4.1 mixed-precision page management (INT8 for rarely used pages).
// The pages fix no scale granularity.  Here every cached (token, kv head) row
// carries one fp32 scale, so quantise-on-append touches only its own slot:
//   amax   = max_j |x_j|
//   scale  = amax / Q            (fp32, rounded once; Q = 127 INT8, 448 E4M3)
//   code_j = INT8: round-half-even(x_j / scale) clamped to [-127, 127]
//            E4M3: x_j / scale (fp32) rounded to the nearest E4M3 value,
//                  ties to even, finite overflow saturating to +-448
// and a row of zeros stores scale 0 and zero codes.  The cached value is
// code_j * scale; decode widens codes to fp32 exactly and applies the K scale
// to each dot product and the V scale to each softmax weight.
//
// Pages: the (block, kv head) page of an 8-bit pool holds the block's
// block_size code rows of head_dim bytes, then ceil(4 * block_size / head_dim)
// rows that start with the rows' fp32 scales (the rest zero), so one
// contiguous copy moves a page with its scales.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

enum { kFmtI8 = PA_I8, kFmtE4M3 = PA_E4M3 };

__host__ __device__ constexpr int q8_scale_rows(int block_size, int head_dim) {
    return (4 * block_size + head_dim - 1) / head_dim;
}
__host__ __device__ constexpr int q8_page_bytes(int block_size, int head_dim) {
    return (block_size + q8_scale_rows(block_size, head_dim)) * head_dim;
}

template <int Fmt> struct Q8;

template <> struct Q8<kFmtI8> {
    static constexpr float kQmax = 127.0f;
    __device__ static inline uint32_t encode(float v) {  // v = x / scale
        int c = __float2int_rn(v);
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        return static_cast<uint32_t>(c) & 0xffu;
    }
    // four codes (one 32-bit word, code i in byte i) -> four exact floats.
    // Byte b = code + 128 is placed as the low mantissa byte of 2^23: the
    // float 2^23 + b, minus 2^23 + 128, is the code itself.
    __device__ static inline void widen4(uint32_t w, float *f) {
        const uint32_t u = w ^ 0x80808080u;
        f[0] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7540)) - 8388736.0f;
        f[1] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7541)) - 8388736.0f;
        f[2] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7542)) - 8388736.0f;
        f[3] = __uint_as_float(__byte_perm(u, 0x4b000000u, 0x7543)) - 8388736.0f;
    }
};

template <> struct Q8<kFmtE4M3> {
    static constexpr float kQmax = 448.0f;
    __device__ static inline uint32_t encode(float v) {
        return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
    }
    // four codes -> four exact floats (every E4M3 value is an fp16 value)
    __device__ static inline void widen4(uint32_t w, float *f) {
        const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
        const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
        f[0] = a.x, f[1] = a.y, f[2] = b.x, f[3] = b.y;
    }
};

// One query / key element of a 16-bit or fp32 row, widened to fp32.
__device__ inline float load_elt(const char *row, int dtype, int j) {
    if (dtype == PA_F32)
        return reinterpret_cast<const float *>(row)[j];
    const uint16_t u = reinterpret_cast<const uint16_t *>(row)[j];
    if (dtype == PA_F16)
        return __half2float(__ushort_as_half(u));
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

}  // namespace pa
