// The 8-bit cache's quantization rule on the device (the quantizing append,
// append_quant.cu).
//
// For a row x of D = 128 activations: scale = max|x| / Qmax and
// code = x / scale rounded to the nearest int8 or E4M3 value (ties to even),
// both divisions in fp32 with round to nearest even, saturated to +-Qmax; an
// all-zero row has scale 0 and zero codes. One warp holds a row, four
// consecutive elements a lane.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

template <typename T>
__device__ __forceinline__ float act_to_f32(T x);
template <>
__device__ __forceinline__ float act_to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float act_to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

// One code of x / s (s > 0).
template <int CODE>
__device__ __forceinline__ uint32_t quant_encode(float x, float s) {
    const float v = __fdiv_rn(x, s);
    if constexpr (CODE == PKV_INT8) {
        int c = __float2int_rn(v);
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        return (uint32_t)(uint8_t)(int8_t)c;
    } else {
        return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
    }
}

// This lane's four elements (8 bytes of T, element 0 first) of a row held by
// the whole warp: the row's scale and this lane's four codes (one 32-bit
// word, element 0 in the low byte).
template <typename T, int CODE>
__device__ __forceinline__ void quantize_lane4(uint2 raw, uint32_t &word_out, float &scale_out) {
    constexpr float kQmax = CODE == PKV_INT8 ? 127.f : 448.f;
    const T *e = reinterpret_cast<const T *>(&raw);
    float x[4], a = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[i] = act_to_f32<T>(e[i]);
        a = fmaxf(a, fabsf(x[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float s = __fdiv_rn(a, kQmax);
    uint32_t word = 0;
    if (a != 0.f) {
#pragma unroll
        for (int i = 0; i < 4; ++i) word |= quant_encode<CODE>(x[i], s) << (8 * i);
    }
    word_out = word;
    scale_out = s;
}

}  // namespace pkv
