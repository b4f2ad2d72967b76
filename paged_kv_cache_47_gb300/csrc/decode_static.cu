// pkv_decode_attention_static: decode attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: a program that
// has already given its whole device-memory budget to the KV-cache pool, a
// plug-in that may only use memory its host framework owns, or code on a path
// where cudaMalloc (which can synchronise the device) is not allowed. For them
// the split-K scratch lives in a fixed array in the library's own device
// memory, declared below. Every GPU that loads the library keeps that array
// for the life of the process.
//
// The array is shared by every call on a device. Its first bytes are the
// split-K arrival counters, which must read zero when a call starts: a
// __device__ array starts zeroed and every call that completes puts the
// counters back to zero, so nothing has to be cleared between calls. A call
// whose kernel gave up on a timed-out wait can leave counters set; the error
// reader then zeroes the array (clear_static_scratch). Two calls whose kernels
// overlap on the GPU (different streams, or unordered graph branches) would
// use the same bytes at the same time and race, so order such calls (for
// example, issue them on one stream).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_pkv_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
int g_scratch_sms[kMaxDevices] = {0};
std::mutex g_scratch_mu;

// Per-device set-up, done by the first call on each device with that device
// current: the device address of the scratch array (host code only sees a
// host-side stand-in for the symbol) and the SM count.
pkv_status scratch_for_current_device(void **ptr, int *sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return pkv::set_last_error(PKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return pkv::set_last_error(PKV_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_pkv_static_scratch);
        if (e != cudaSuccess)
            return pkv::set_last_error(PKV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                                       cudaGetErrorString(e));
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return pkv::set_last_error(PKV_ERR_CUDA, "querying the SM count: %s",
                                       cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
        g_scratch_sms[dev] = n;
    }
    *ptr = g_scratch_ptr[dev];
    *sms = g_scratch_sms[dev];
    return PKV_OK;
}

}  // namespace

namespace pkv {
// Zero the scratch array of the current device if a call has used it there.
// The memset is ordered on `stream` and waited for before returning, so it is
// complete whatever stream the caller uses next (a plain cudaMemset would be
// asynchronous for device memory and ordered only against the legacy default
// stream, which non-blocking streams do not synchronise with).
cudaError_t clear_static_scratch(cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        p = g_scratch_ptr[dev];
    }
    if (!p) return cudaSuccess;
    e = cudaMemsetAsync(p, 0, PKV_STATIC_SCRATCH_BYTES, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}
}  // namespace pkv

extern "C" pkv_status pkv_decode_attention_static(
    const pkv_cache_desc *cache, const void *q, int32_t num_seqs, int32_t num_q_heads,
    const void *k_pool, const void *v_pool, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *context_lens, float scale, void *out,
    int32_t out_dtype, void *stream) {
    void *scratch = nullptr;
    int sms = 0;
    pkv_status st = scratch_for_current_device(&scratch, &sms);
    if (st != PKV_OK) return st;
    // one split-K CTA per SM; the scratch this needs depends only on the
    // SM count, the q heads per kv head and head_dim
    const size_t need = pkv_decode_workspace_bytes_ex(cache, num_q_heads, sms);
    if (need == 0)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG,
                                   "invalid cache descriptor or head counts");
    if (need > PKV_STATIC_SCRATCH_BYTES)
        return pkv::set_last_error(
            PKV_ERR_WORKSPACE,
            "this shape needs %zu bytes of split-K scratch; the fixed scratch holds %u bytes "
            "(use pkv_decode_attention with a workspace)",
            need, (unsigned)PKV_STATIC_SCRATCH_BYTES);
    pkv_decode_options opts = {};
    opts.num_ctas = sms;
    return pkv_decode_attention_ex(cache, q, num_seqs, num_q_heads, k_pool, v_pool, block_tables,
                                   max_blocks_per_seq, context_lens, scale, out, out_dtype,
                                   scratch, PKV_STATIC_SCRATCH_BYTES, stream, &opts);
}
