// KV append (slot write) and whole-block copy kernels.
//
// Append: each new token's K and V rows go to their slot, slot = block * B +
// offset ("KV-Cache Optimization & PagedAttention for Long-Context Agents",
// section "Key KV-Cache Optimization Principles", item 1). Block copy: the one
// block a writer hits while others still share it is duplicated
// ("PagedAttention — Math + Memory Model", section "Copy-on-write").
//
// Both are pure byte movement with 16-byte vector loads and stores, coalesced
// along head_dim; one thread moves one 16-byte vector of K and the matching
// vector of V.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {

// Programmatic dependent launch (see device_utils.cuh; duplicated here to keep
// this translation unit free of the decode headers).
__device__ __forceinline__ void append_wait_prior_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void append_allow_next_grid() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Slot of token i: slot_mapping[i], or (slot_mapping NULL: the token is the
// newest of sequence i) the block table's slot of position L - 1, -1 for an
// empty context. A length past the table is clamped as the decode clamps it,
// and a block id outside the pool is skipped (the decode flags both).
__device__ __forceinline__ int64_t append_slot(const int64_t *slot_mapping, const int32_t *tables,
                                               const int32_t *lens, int M, int B, int NB,
                                               int tok) {
    if (slot_mapping) return __ldg(slot_mapping + tok);
    int L = __ldg(lens + tok);
    if (L > M * B) L = M * B;
    if (L <= 0) return -1;
    const int blk = __ldg(tables + (size_t)tok * M + (L - 1) / B);
    if (blk < 0 || blk >= NB) return -1;
    return (int64_t)blk * B + (L - 1) % B;
}

// grid-stride over (token, vector-in-token); vectors per token = Hk*D*es/16.
// With inputs_ready each thread reads its first vector (slot, K and V) before
// the wait on the previous kernel, so only the stores remain after it.
__global__ void __launch_bounds__(256) append_kernel(const uint4 *__restrict__ k_new,
                                                     const uint4 *__restrict__ v_new,
                                                     const int64_t *__restrict__ slot_mapping,
                                                     const int32_t *__restrict__ tables,
                                                     const int32_t *__restrict__ lens, int M,
                                                     int num_tokens, uint4 *__restrict__ k_pool,
                                                     uint4 *__restrict__ v_pool, int NB, int B,
                                                     int vec_per_row, int vec_per_token,
                                                     int inputs_ready, unsigned *err) {
    // launched with programmatic serialisation: the previous kernel on the
    // stream must be complete before any pool byte is touched; the next one
    // (the decode) may be scheduled meanwhile
    append_allow_next_grid();
    const int64_t total = (int64_t)num_tokens * vec_per_token;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    int64_t slot = -1;
    uint4 kv = {}, vv = {};
    const bool early = inputs_ready && i < total;
    if (early) {
        slot = append_slot(slot_mapping, tables, lens, M, B, NB, (int)(i / vec_per_token));
        kv = __ldg(k_new + i);
        vv = __ldg(v_new + i);
    }
    append_wait_prior_grid();
    for (bool have = early; i < total; i += stride, have = false) {
        const int tok = (int)(i / vec_per_token);
        const int v = (int)(i - (int64_t)tok * vec_per_token);
        if (!have) slot = append_slot(slot_mapping, tables, lens, M, B, NB, tok);
        if (slot < 0) continue;
        const int64_t blk = slot / B;
        const int off = (int)(slot - blk * B);
        if (blk >= NB) {
            if (v == 0) atomicOr(err, PKV_DEVERR_SLOT);
            continue;
        }
        if (!have) {
            kv = __ldg(k_new + i);
            vv = __ldg(v_new + i);
        }
        const int g = v / vec_per_row;
        const int w = v - g * vec_per_row;
        const int Hk = vec_per_token / vec_per_row;
        const int64_t dst = ((blk * Hk + g) * B + off) * (int64_t)vec_per_row + w;
        k_pool[dst] = kv;
        v_pool[dst] = vv;
    }
}

cudaError_t launch_append(int dtype, const void *k_new, const void *v_new,
                          const int64_t *slot_mapping, int num_tokens, void *k_pool, void *v_pool,
                          int NB, int Hk, int B, int D, int inputs_ready, unsigned *err,
                          cudaStream_t st, const int32_t *tables, const int32_t *lens, int M) {
    const int es = dtype == PKV_F32 ? 4 : 2;
    const int vec_per_row = D * es / 16;
    const int vec_per_token = Hk * vec_per_row;
    const int64_t total = (int64_t)num_tokens * vec_per_token;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_kernel, static_cast<const uint4 *>(k_new),
                              static_cast<const uint4 *>(v_new), slot_mapping, tables, lens, M,
                              num_tokens,
                              static_cast<uint4 *>(k_pool), static_cast<uint4 *>(v_pool), NB, B,
                              vec_per_row, vec_per_token, inputs_ready, err);
}

// blockIdx.y = pair; grid-stride over the block's 16-byte vectors.
__global__ void __launch_bounds__(256) block_copy_kernel(const CopyPairs pairs, uint4 *k_pool,
                                                         uint4 *v_pool, int64_t vec_per_block) {
    const int pr = blockIdx.y;
    const int64_t src = pairs.src[pr] * vec_per_block;
    const int64_t dst = pairs.dst[pr] * vec_per_block;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < vec_per_block;
         i += (int64_t)gridDim.x * blockDim.x) {
        k_pool[dst + i] = k_pool[src + i];
        v_pool[dst + i] = v_pool[src + i];
    }
}

cudaError_t launch_block_copy(const CopyPairs &pairs, int n, void *k_pool, void *v_pool,
                              size_t block_bytes, cudaStream_t st) {
    const int64_t vec = (int64_t)(block_bytes / 16);
    const int threads = 256;
    int64_t bx = (vec + threads * 4 - 1) / (threads * 4);
    if (bx < 1) bx = 1;
    if (bx > 1024) bx = 1024;
    dim3 grid((unsigned)bx, (unsigned)n);
    block_copy_kernel<<<grid, threads, 0, st>>>(pairs, static_cast<uint4 *>(k_pool),
                                                static_cast<uint4 *>(v_pool), vec);
    return cudaGetLastError();
}

}  // namespace pkv
