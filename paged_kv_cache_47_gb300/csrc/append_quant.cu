// Quantized KV append: each new token's K and V rows become 8-bit codes with
// one fp32 scale per (token, kv head) row, written at their slot.
//
// The pages name an 8-bit KV cache as the lever that halves each decode's
// read ("Contiguous vs Paged KV Cache on RDNA4", section "The order of the
// memory levers"); the format (include/pkv.h, "8-bit KV cache") is this
// library's reading: scale = max|x| / Qmax and code = x / scale rounded to
// the nearest int8 or E4M3 value (ties to even), both divisions in fp32 with
// round to nearest even, saturated to +-Qmax; an all-zero row has scale 0.
//
// One warp per (token, kv head) row of D = 128 activations: each lane holds
// four consecutive elements (one 8-byte load), the row maximum is a warp
// max-reduction, and the lane writes its four codes as one 32-bit store.
// With inputs_ready (pkv_append_quant_ex) a warp loads and quantizes its
// first row before it waits for the preceding kernel; only stores follow.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"
#include "quant_codec.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ void wait_prior_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_next_grid() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The row `src` (D = 128 elements of T) quantized: this lane's four codes
// (one 32-bit word) and the row's scale.
template <typename T, int CODE>
__device__ __forceinline__ void quantize_row(const T *__restrict__ src, uint32_t &word_out,
                                             float &scale_out, int lane) {
    quantize_lane4<T, CODE>(__ldg(reinterpret_cast<const uint2 *>(src) + lane), word_out,
                            scale_out);
}

// One (token, kv head) row quantized, waiting to be stored.
struct QRow {
    int64_t row = -1;      // row of the pools; -1: nothing to store
    uint32_t kw = 0, vw = 0;
    float ks = 0.f, vs = 0.f;
};

// The slot of token tok: slots[tok], or (slots NULL) position lens[tok] - 1
// of table row tok (-1 for an empty context or a block id outside the pool,
// which the decode flags).
__device__ __forceinline__ int64_t token_slot(const int64_t *slots, const int32_t *tables,
                                              const int32_t *lens, int M, int B, int NB, int tok) {
    if (slots) return __ldg(slots + tok);
    int L = __ldg(lens + tok);
    if (L > M * B) L = M * B;
    if (L <= 0) return -1;
    const int blk = __ldg(tables + (size_t)tok * M + (L - 1) / B);
    if (blk < 0 || blk >= NB) return -1;
    return (int64_t)blk * B + (L - 1) % B;
}

template <typename T, int CODE>
__device__ __forceinline__ QRow quantize_token_row(const T *__restrict__ k_new,
                                                   const T *__restrict__ v_new,
                                                   const int64_t *__restrict__ slots,
                                                   const int32_t *tables, const int32_t *lens,
                                                   int M, int64_t r, int NB, int Hk, int B,
                                                   unsigned *err, int lane) {
    constexpr int D = 128;
    QRow q;
    const int tok = (int)(r / Hk), g = (int)(r - (int64_t)tok * Hk);
    const int64_t slot = token_slot(slots, tables, lens, M, B, NB, tok);
    if (slot < 0) return q;
    const int64_t blk = slot / B;
    const int off = (int)(slot - blk * B);
    if (blk >= NB) {
        if (lane == 0 && g == 0) atomicOr(err, PKV_DEVERR_SLOT);
        return q;
    }
    q.row = (blk * Hk + g) * B + off;
    quantize_row<T, CODE>(k_new + r * D, q.kw, q.ks, lane);
    quantize_row<T, CODE>(v_new + r * D, q.vw, q.vs, lane);
    return q;
}

__device__ __forceinline__ void store_row(const QRow &q, uint8_t *__restrict__ k_codes,
                                          uint8_t *__restrict__ v_codes,
                                          float *__restrict__ k_scales,
                                          float *__restrict__ v_scales, int lane) {
    constexpr int D = 128;
    if (q.row < 0) return;
    reinterpret_cast<uint32_t *>(k_codes + q.row * D)[lane] = q.kw;
    reinterpret_cast<uint32_t *>(v_codes + q.row * D)[lane] = q.vw;
    if (lane == 0) {
        k_scales[q.row] = q.ks;
        v_scales[q.row] = q.vs;
    }
}

// grid-stride over rows (token, kv head); one warp per row. With
// inputs_ready each warp reads and quantizes its first row before the wait
// on the previous kernel, so only its stores remain after it.
template <typename T, int CODE>
__global__ void __launch_bounds__(256) append_quant_kernel(
    const T *__restrict__ k_new, const T *__restrict__ v_new, const int64_t *__restrict__ slots,
    const int32_t *__restrict__ tables, const int32_t *__restrict__ lens, int M, int num_tokens,
    uint8_t *__restrict__ k_codes, uint8_t *__restrict__ v_codes, float *__restrict__ k_scales,
    float *__restrict__ v_scales, int NB, int Hk, int B, int inputs_ready, unsigned *err) {
    // programmatic serialisation: the previous kernel on the stream completes
    // before any pool byte is touched; the next one may be scheduled meanwhile
    allow_next_grid();
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)num_tokens * Hk;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    QRow first;
    const bool early = inputs_ready && r < rows;
    if (early)
        first = quantize_token_row<T, CODE>(k_new, v_new, slots, tables, lens, M, r, NB, Hk, B, err,
                                            lane);
    wait_prior_grid();
    for (bool have = early; r < rows; r += warps, have = false) {
        const QRow q =
            have ? first
                 : quantize_token_row<T, CODE>(k_new, v_new, slots, tables, lens, M, r, NB, Hk, B,
                                               err, lane);
        store_row(q, k_codes, v_codes, k_scales, v_scales, lane);
    }
}

template <typename T, int CODE>
cudaError_t launch(const void *k_new, const void *v_new, const int64_t *slots,
                   const int32_t *tables, const int32_t *lens, int M, int num_tokens,
                   void *k_codes, void *v_codes, float *k_scales, float *v_scales, int NB, int Hk,
                   int B, int inputs_ready, unsigned *err, cudaStream_t st) {
    const int64_t rows = (int64_t)num_tokens * Hk;
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_quant_kernel<T, CODE>, static_cast<const T *>(k_new),
                              static_cast<const T *>(v_new), slots, tables, lens, M, num_tokens,
                              static_cast<uint8_t *>(k_codes), static_cast<uint8_t *>(v_codes),
                              k_scales, v_scales, NB, Hk, B, inputs_ready, err);
}

}  // namespace

cudaError_t launch_append_quant(int code_dtype, int act_dtype, const void *k_new,
                                const void *v_new, const int64_t *slots, int num_tokens,
                                void *k_codes, void *v_codes, float *k_scales, float *v_scales,
                                int NB, int Hk, int B, int inputs_ready, unsigned *err,
                                cudaStream_t st, const int32_t *tables, const int32_t *lens,
                                int M) {
    auto *L = act_dtype == PKV_F16
                  ? (code_dtype == PKV_INT8 ? &launch<__half, PKV_INT8> : &launch<__half, PKV_FP8_E4M3>)
                  : (code_dtype == PKV_INT8 ? &launch<__nv_bfloat16, PKV_INT8>
                                            : &launch<__nv_bfloat16, PKV_FP8_E4M3>);
    return L(k_new, v_new, slots, tables, lens, M, num_tokens, k_codes, v_codes, k_scales,
             v_scales, NB, Hk, B, inputs_ready, err, st);
}

}  // namespace pkv
