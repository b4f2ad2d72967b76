// Flat spans: a KV cache kept contiguous in virtual memory (include/pkv_flat.h).
//
// Passage: each sequence reserves one flat virtual range and physical memory
// is committed into it on demand, so the attention kernel reads a flat span
// instead of gathering through a block table ("Contiguous vs Paged KV Cache
// on RDNA4", section "Why the single-user verdict flipped", on vAttention).
//
// GB300 form: one virtual reservation (cuMemAddressReserve) for all slots;
// each slot's K and V spans grow by mapping granularity-sized physical chunks
// (cuMemCreate + cuMemMap + cuMemSetAccess). The driver calls are resolved
// once through the runtime's driver entry points, so the library does not
// link the driver directly. A device array of committed tokens per slot is
// kept in step with the mappings and bounds every device access.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <new>
#include <vector>

#include "../../include/pkv_flat.h"
#include "pkv_internal.h"

namespace {

// ---------------------------------------------------------------- driver calls
struct Driver {
    CUresult (*mem_address_reserve)(CUdeviceptr *, size_t, size_t, CUdeviceptr, unsigned long long);
    CUresult (*mem_address_free)(CUdeviceptr, size_t);
    CUresult (*mem_create)(CUmemGenericAllocationHandle *, size_t, const CUmemAllocationProp *,
                           unsigned long long);
    CUresult (*mem_release)(CUmemGenericAllocationHandle);
    CUresult (*mem_map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle,
                        unsigned long long);
    CUresult (*mem_unmap)(CUdeviceptr, size_t);
    CUresult (*mem_set_access)(CUdeviceptr, size_t, const CUmemAccessDesc *, size_t);
    CUresult (*mem_get_granularity)(size_t *, const CUmemAllocationProp *,
                                    CUmemAllocationGranularity_flags);
    bool ok = false;
};

template <typename F>
bool resolve(const char *name, F &fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return false;
    fn = reinterpret_cast<F>(p);
    return true;
}

const Driver &driver() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        d.ok = resolve("cuMemAddressReserve", d.mem_address_reserve) &&
               resolve("cuMemAddressFree", d.mem_address_free) &&
               resolve("cuMemCreate", d.mem_create) && resolve("cuMemRelease", d.mem_release) &&
               resolve("cuMemMap", d.mem_map) && resolve("cuMemUnmap", d.mem_unmap) &&
               resolve("cuMemSetAccess", d.mem_set_access) &&
               resolve("cuMemGetAllocationGranularity", d.mem_get_granularity);
    });
    return d;
}

pkv_status fail_cu(CUresult r, const char *what) {
    return pkv::set_last_error(PKV_ERR_CUDA, "%s failed (CUresult %d)", what, (int)r);
}

pkv_status fail_rt(cudaError_t e, const char *what) {
    return pkv::set_last_error(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- append kernel
// grid-stride over (token, 16-byte vector of its Hk rows)
__global__ void __launch_bounds__(256) flat_append_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int32_t *__restrict__ slots, const int32_t *__restrict__ positions, int num_tokens,
    uint8_t *k_base, size_t slot_stride, size_t v_off, const int32_t *__restrict__ committed,
    int num_slots, int vec_per_token, unsigned *err) {
    // programmatic serialisation: the previous kernel completes before the
    // spans are written; the next one may be scheduled meanwhile
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t total = (int64_t)num_tokens * vec_per_token;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int tok = (int)(i / vec_per_token);
        const int v = (int)(i - (int64_t)tok * vec_per_token);
        const int slot = __ldg(slots + tok), pos = __ldg(positions + tok);
        if (slot < 0 || slot >= num_slots || pos < 0 || pos >= __ldg(committed + slot)) {
            if (v == 0) atomicOr(err, PKV_DEVERR_SLOT);
            continue;
        }
        // token-major span: the token's Hk rows are adjacent
        uint4 *dst = reinterpret_cast<uint4 *>(k_base + (size_t)slot * slot_stride) +
                     (size_t)pos * vec_per_token + v;
        dst[0] = __ldg(k_new + i);
        *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(dst) + v_off) = __ldg(v_new + i);
    }
}

}  // namespace

struct pkv_flat_cache {
    int device = 0;
    int32_t num_slots = 0, capacity = 0, Hk = 0, D = 0, dtype = 0;
    size_t token_bytes = 0;     // Hk * D * element bytes
    size_t gran = 0, region = 0, slot_stride = 0;
    CUdeviceptr va = 0;
    size_t va_size = 0;
    std::vector<std::vector<CUmemGenericAllocationHandle>> chunks;   // per slot, K then V pairs
    std::vector<int32_t> committed;                                    // host copy
    int32_t *committed_dev = nullptr;
    size_t committed_bytes = 0;
    std::mutex mu;

    CUmemAllocationProp prop() const {
        CUmemAllocationProp p = {};
        p.type = CU_MEM_ALLOCATION_TYPE_PINNED;
        p.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
        p.location.id = device;
        return p;
    }

    // Unmap and release every chunk of slot (lock held).
    pkv_status release_locked(int32_t slot) {
        const Driver &d = driver();
        if (committed[slot] != 0) {
            const int32_t zero = 0;
            cudaError_t e = cudaMemcpy(committed_dev + slot, &zero, 4, cudaMemcpyHostToDevice);
            if (e != cudaSuccess) return fail_rt(e, "cudaMemcpy(committed tokens)");
            committed[slot] = 0;
        }
        std::vector<CUmemGenericAllocationHandle> &c = chunks[slot];
        const size_t n = c.size() / 2;
        const CUdeviceptr base = va + (size_t)slot * slot_stride;
        for (size_t i = 0; i < n; ++i) {
            CUresult r = d.mem_unmap(base + i * gran, gran);
            if (r == CUDA_SUCCESS) r = d.mem_unmap(base + region + i * gran, gran);
            if (r != CUDA_SUCCESS) return fail_cu(r, "cuMemUnmap");
        }
        for (CUmemGenericAllocationHandle h : c) {
            CUresult r = d.mem_release(h);
            if (r != CUDA_SUCCESS) return fail_cu(r, "cuMemRelease");
        }
        committed_bytes -= c.size() * gran;
        c.clear();
        return PKV_OK;
    }
};

extern "C" {

pkv_status pkv_flat_create(int32_t num_slots, int32_t capacity_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int32_t dtype, pkv_flat_cache **out) {
    if (!out) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (num_slots < 1 || capacity_tokens < pkv::kFlatRowsPerGroup ||
        capacity_tokens % pkv::kFlatRowsPerGroup != 0 || num_kv_heads < 1)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG,
                                   "num_slots >= 1, capacity a positive multiple of %d, "
                                   "num_kv_heads >= 1", pkv::kFlatRowsPerGroup);
    if (head_dim != 64 && head_dim != 128)
        return pkv::set_last_error(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (dtype != PKV_F16 && dtype != PKV_BF16)
        return pkv::set_last_error(PKV_ERR_UNSUPPORTED, "dtype %d (supported: PKV_F16, PKV_BF16)",
                                   dtype);
    const Driver &d = driver();
    if (!d.ok)
        return pkv::set_last_error(PKV_ERR_UNSUPPORTED, "virtual memory calls are not available");
    pkv_flat_cache *fc = new (std::nothrow) pkv_flat_cache();
    if (!fc) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "out of host memory");
    cudaError_t e = cudaGetDevice(&fc->device);
    if (e == cudaSuccess) e = cudaFree(nullptr);   // make the device's context current
    if (e != cudaSuccess) {
        delete fc;
        return fail_rt(e, "device set-up");
    }
    fc->num_slots = num_slots;
    fc->capacity = capacity_tokens;
    fc->Hk = num_kv_heads;
    fc->D = head_dim;
    fc->dtype = dtype;
    fc->token_bytes = (size_t)num_kv_heads * head_dim * 2;
    const CUmemAllocationProp pr = fc->prop();
    CUresult r = d.mem_get_granularity(&fc->gran, &pr, CU_MEM_ALLOC_GRANULARITY_MINIMUM);
    if (r != CUDA_SUCCESS) {
        delete fc;
        return fail_cu(r, "cuMemGetAllocationGranularity");
    }
    const size_t span = (size_t)capacity_tokens * fc->token_bytes;
    fc->region = (span + fc->gran - 1) / fc->gran * fc->gran;
    fc->slot_stride = 2 * fc->region;
    fc->va_size = fc->slot_stride * (size_t)num_slots;
    r = d.mem_address_reserve(&fc->va, fc->va_size, fc->gran, 0, 0);
    if (r != CUDA_SUCCESS) {
        delete fc;
        return fail_cu(r, "cuMemAddressReserve");
    }
    fc->chunks.resize(num_slots);
    fc->committed.assign(num_slots, 0);
    e = cudaMalloc(&fc->committed_dev, sizeof(int32_t) * num_slots);
    if (e == cudaSuccess) e = cudaMemset(fc->committed_dev, 0, sizeof(int32_t) * num_slots);
    if (e != cudaSuccess) {
        if (fc->committed_dev) cudaFree(fc->committed_dev);
        d.mem_address_free(fc->va, fc->va_size);
        delete fc;
        return fail_rt(e, "committed-token array");
    }
    *out = fc;
    return PKV_OK;
}

void pkv_flat_destroy(pkv_flat_cache *fc) {
    if (!fc) return;
    {
        std::lock_guard<std::mutex> lk(fc->mu);
        for (int32_t s = 0; s < fc->num_slots; ++s) fc->release_locked(s);
        driver().mem_address_free(fc->va, fc->va_size);
        cudaFree(fc->committed_dev);
    }
    delete fc;
}

pkv_status pkv_flat_reserve(pkv_flat_cache *fc, int32_t slot, int32_t tokens) {
    if (!fc) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "cache is NULL");
    if (slot < 0 || slot >= fc->num_slots || tokens < 0 || tokens > fc->capacity)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "slot %d / tokens %d out of range", slot,
                                   tokens);
    std::lock_guard<std::mutex> lk(fc->mu);
    if (tokens <= fc->committed[slot]) return PKV_OK;
    const Driver &d = driver();
    const CUmemAllocationProp pr = fc->prop();
    CUmemAccessDesc acc = {};
    acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    acc.location.id = fc->device;
    acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    std::vector<CUmemGenericAllocationHandle> &c = fc->chunks[slot];
    const size_t need = ((size_t)tokens * fc->token_bytes + fc->gran - 1) / fc->gran;
    const CUdeviceptr base = fc->va + (size_t)slot * fc->slot_stride;
    while (c.size() / 2 < need) {
        const size_t i = c.size() / 2;
        for (int kv = 0; kv < 2; ++kv) {
            const CUdeviceptr at = base + (kv ? fc->region : 0) + i * fc->gran;
            CUmemGenericAllocationHandle h;
            CUresult r = d.mem_create(&h, fc->gran, &pr, 0);
            if (r != CUDA_SUCCESS) return fail_cu(r, "cuMemCreate");
            r = d.mem_map(at, fc->gran, 0, h, 0);
            if (r == CUDA_SUCCESS) r = d.mem_set_access(at, fc->gran, &acc, 1);
            if (r != CUDA_SUCCESS) {
                d.mem_unmap(at, fc->gran);
                d.mem_release(h);
                // keep K and V chunk counts equal: undo a lone K chunk
                if (kv == 1) {
                    d.mem_unmap(base + i * fc->gran, fc->gran);
                    d.mem_release(c.back());
                    c.pop_back();
                    fc->committed_bytes -= fc->gran;
                }
                return fail_cu(r, "cuMemMap / cuMemSetAccess");
            }
            c.push_back(h);
            fc->committed_bytes += fc->gran;
        }
    }
    const size_t held = c.size() / 2 * fc->gran / fc->token_bytes;
    const int32_t now = (int32_t)(held < (size_t)fc->capacity ? held : (size_t)fc->capacity);
    cudaError_t e = cudaMemcpy(fc->committed_dev + slot, &now, 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_rt(e, "cudaMemcpy(committed tokens)");
    fc->committed[slot] = now;
    return PKV_OK;
}

pkv_status pkv_flat_release(pkv_flat_cache *fc, int32_t slot) {
    if (!fc) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "cache is NULL");
    if (slot < 0 || slot >= fc->num_slots)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "slot %d out of range", slot);
    std::lock_guard<std::mutex> lk(fc->mu);
    return fc->release_locked(slot);
}

pkv_status pkv_flat_get_info(pkv_flat_cache *fc, pkv_flat_info *out) {
    if (!fc || !out) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "NULL argument");
    std::lock_guard<std::mutex> lk(fc->mu);
    out->k_base = reinterpret_cast<void *>(fc->va);
    out->slot_stride = fc->slot_stride;
    out->v_offset = fc->region;
    out->granularity = fc->gran;
    out->committed_bytes = fc->committed_bytes;
    out->committed_tokens = fc->committed_dev;
    return PKV_OK;
}

pkv_status pkv_flat_append(pkv_flat_cache *fc, const void *k_new, const void *v_new,
                           const int32_t *slots, const int32_t *positions, int32_t num_tokens,
                           void *stream) {
    if (!fc) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "cache is NULL");
    if (num_tokens < 0) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slots || !positions)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) % 16 ||
        (reinterpret_cast<uintptr_t>(slots) | reinterpret_cast<uintptr_t>(positions)) % 4)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "misaligned pointer");
    unsigned *err = nullptr;
    pkv_status st = pkv::device_error_word(&err);
    if (st != PKV_OK) return st;
    const int vec_per_token = (int)(fc->token_bytes / 16);
    const int64_t total = (int64_t)num_tokens * vec_per_token;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, flat_append_kernel, static_cast<const uint4 *>(k_new),
                                       static_cast<const uint4 *>(v_new), slots, positions,
                                       num_tokens, reinterpret_cast<uint8_t *>(fc->va),
                                       fc->slot_stride, fc->region,
                                       (const int32_t *)fc->committed_dev, fc->num_slots,
                                       vec_per_token, err);
    if (e != cudaSuccess) return fail_rt(e, "flat append launch");
    return PKV_OK;
}

size_t pkv_flat_decode_workspace_bytes(pkv_flat_cache *fc, int32_t num_q_heads, int32_t num_ctas) {
    if (!fc) return 0;
    pkv::FlatGeom g{reinterpret_cast<void *>(fc->va), fc->slot_stride, fc->region,
                    fc->committed_dev, fc->num_slots, fc->capacity, fc->Hk, fc->D, fc->dtype};
    return pkv::flat_workspace_bytes(g, num_q_heads, num_ctas);
}

pkv_status pkv_decode_attention_flat(pkv_flat_cache *fc, const void *q, int32_t num_seqs,
                                     int32_t num_q_heads, const int32_t *slots,
                                     const int32_t *context_lens, float scale, void *out,
                                     int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                     void *stream, const pkv_decode_options *options) {
    if (!fc) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "cache is NULL");
    pkv::FlatGeom g{reinterpret_cast<void *>(fc->va), fc->slot_stride, fc->region,
                    fc->committed_dev, fc->num_slots, fc->capacity, fc->Hk, fc->D, fc->dtype};
    return pkv::decode_flat(g, q, num_seqs, num_q_heads, slots, context_lens, scale, out,
                            out_dtype, workspace, workspace_bytes,
                            static_cast<cudaStream_t>(stream), options);
}

}  // extern "C"
