// The C ABI of libpkv (include/pkv.h): argument checks, kernel dispatch and
// the device error word.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <memory>
#include <mutex>
#include <unordered_set>
#include <vector>

#include "../../include/pkv.h"
#include "decomp.h"
#include "pkv_internal.h"

namespace {

// ---------------------------------------------------------------- errors
thread_local char g_msg[512] = "";

pkv_status fail(pkv_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

pkv_status cuda_fail(cudaError_t e, const char *what) {
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One error word per device, in the library's own static device memory.
__device__ unsigned int g_pkv_error_word;

constexpr int kMaxDevices = 64;
unsigned *g_err_ptr[kMaxDevices] = {nullptr};
std::mutex g_err_mu;

pkv_status device_error_ptr(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_pkv_error_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        g_err_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_err_ptr[dev];
    return PKV_OK;
}

// ---------------------------------------------------------------- checks
int elem_bytes(int dtype) { return dtype == PKV_F32 ? 4 : 2; }
bool valid_dtype(int dtype) { return dtype == PKV_F32 || dtype == PKV_F16 || dtype == PKV_BF16; }
bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pkv_status check_cache(const pkv_cache_desc *c) {
    if (!c) return fail(PKV_ERR_INVALID_ARG, "cache descriptor is NULL");
    if (!valid_dtype(c->dtype)) return fail(PKV_ERR_UNSUPPORTED, "dtype %d", c->dtype);
    if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32)
        return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", c->block_size);
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", c->head_dim);
    if (c->num_kv_heads < 1) return fail(PKV_ERR_INVALID_ARG, "num_kv_heads %d", c->num_kv_heads);
    if (c->num_blocks < 1) return fail(PKV_ERR_INVALID_ARG, "num_blocks %d", c->num_blocks);
    return PKV_OK;
}

pkv_status check_qcache(const pkv_qcache_desc *c) {
    if (!c) return fail(PKV_ERR_INVALID_ARG, "cache descriptor is NULL");
    if (c->code_dtype != PKV_INT8 && c->code_dtype != PKV_FP8_E4M3)
        return fail(PKV_ERR_UNSUPPORTED, "code_dtype %d (supported: PKV_INT8, PKV_FP8_E4M3)",
                    c->code_dtype);
    if (c->act_dtype != PKV_F16 && c->act_dtype != PKV_BF16)
        return fail(PKV_ERR_UNSUPPORTED, "act_dtype %d (supported: PKV_F16, PKV_BF16)", c->act_dtype);
    if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32)
        return fail(PKV_ERR_UNSUPPORTED, "block_size %d (supported: 8, 16, 32)", c->block_size);
    if (c->head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (8-bit caches support 128)", c->head_dim);
    if (c->num_kv_heads < 1) return fail(PKV_ERR_INVALID_ARG, "num_kv_heads %d", c->num_kv_heads);
    if (c->num_blocks < 1) return fail(PKV_ERR_INVALID_ARG, "num_blocks %d", c->num_blocks);
    return PKV_OK;
}

// ---------------------------------------------------------------- decode plan
struct Plan {
    int G, GC, NC, U;
    bool mma;
    int gmax;
    const pkv::DecodeVariant *variant;
    int slots = 2;   // partial slots per CTA: 2 per section of the work list
};

// Head grouping and math path shared by every decode entry point.
pkv_status plan_groups(int Hk, int Hq, const pkv_decode_options *o, bool half, Plan *pl) {
    if (Hq < 1 || Hq % Hk != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d",
                    Hq, Hk);
    const int consumer = o ? o->consumer : 0;
    if (consumer < 0 || consumer > 2) return fail(PKV_ERR_INVALID_ARG, "consumer %d", consumer);
    pl->G = Hq / Hk;
    pl->GC = pl->G < pkv::kMaxHeadsPerUnit ? pl->G : pkv::kMaxHeadsPerUnit;
    pl->NC = (pl->G + pl->GC - 1) / pl->GC;
    pl->U = Hk * pl->NC;
    if (consumer == 2 && !half)
        return fail(PKV_ERR_UNSUPPORTED, "tensor-core math needs fp16 or bf16 K/V");
    // 16-bit K/V go to the tensor cores whatever the group size: with one
    // query head per KV head the SIMT path spends its time converting and
    // reducing, the mma path (query heads padded to n = 8) stays HBM-bound
    pl->mma = half && consumer != 1;
    if (pl->mma) {
        pl->gmax = pl->GC <= 8 ? 8 : 16;
    } else {
        int g = 1;
        while (g < pl->GC) g <<= 1;
        pl->gmax = g;
    }
    return PKV_OK;
}

pkv_status make_plan(const pkv_cache_desc *c, int Hq, const pkv_decode_options *o, Plan *pl) {
    pkv_status st = plan_groups(c->num_kv_heads, Hq, o, c->dtype != PKV_F32, pl);
    if (st != PKV_OK) return st;
    const int D = c->head_dim;
    pl->variant = c->dtype == PKV_F32   ? pkv::find_variant_f32(D, pl->gmax, pl->mma)
                  : c->dtype == PKV_F16 ? pkv::find_variant_f16(D, pl->gmax, pl->mma)
                                        : pkv::find_variant_bf16(D, pl->gmax, pl->mma);
    if (!pl->variant) return fail(PKV_ERR_UNSUPPORTED, "no kernel variant for this shape");
    return PKV_OK;
}

pkv_status make_plan_quant(const pkv_qcache_desc *c, int Hq, const pkv_decode_options *o,
                           Plan *pl) {
    if (o && o->consumer == 1)
        return fail(PKV_ERR_UNSUPPORTED, "8-bit caches use the tensor-core math (consumer 1 given)");
    pkv_status st = plan_groups(c->num_kv_heads, Hq, o, true, pl);
    if (st != PKV_OK) return st;
    // E4M3 units of up to 4 heads: the tensor-core variant sized for 4
    if (c->code_dtype == PKV_FP8_E4M3 && pl->GC <= 4) pl->gmax = 4;
    pl->variant = pkv::find_variant_quant(c->code_dtype, c->act_dtype, c->head_dim, pl->gmax);
    if (!pl->variant) return fail(PKV_ERR_UNSUPPORTED, "no kernel variant for this shape");
    return PKV_OK;
}

// SM count of the current device (queried once per device)
pkv_status sm_count(int *sms) {
    // atomics: first calls from several host threads may race to fill it
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(PKV_ERR_UNSUPPORTED, "device index %d", dev);
    int n = cached[dev].load(std::memory_order_acquire);
    if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "querying the SM count");
        cached[dev].store(n, std::memory_order_release);
    }
    *sms = n;
    return PKV_OK;
}

pkv_status default_ctas(const Plan &pl, int *C) {
    int sms = 0;
    pkv_status st = sm_count(&sms);
    if (st != PKV_OK) return st;
    int occ = pl.variant->max_ctas_per_sm();
    if (occ < 1) return fail(PKV_ERR_CUDA, "split-K kernel cannot be resident (occupancy 0)");
    if (occ > pkv::kMaxCtasPerSm) occ = pkv::kMaxCtasPerSm;
    *C = sms * occ;
    return PKV_OK;
}

// workspace: [PKV_MAX_DECODE_CTAS][4] arrival counters (a fixed region, so
// that no launch's partials ever land where a launch with more CTAs keeps its
// counters), then [C][2][GC][D] partial outputs, then [C][2][4][GC] partial
// log2-sum-exp2 values (one copy per math warp)
constexpr size_t kCounterBytes = (size_t)PKV_MAX_DECODE_CTAS * pkv::kMergeSlices * sizeof(unsigned);
size_t workspace_for(int C, int GC, int D) {
    const size_t W = pkv::kMergeSlices;
    return kCounterBytes + (size_t)C * 2 * GC * (D + W) * sizeof(float);
}

pkv_status max_default_ctas(int *C) {
    int sms = 0;
    pkv_status st = sm_count(&sms);
    if (st != PKV_OK) return st;
    *C = sms * pkv::kMaxCtasPerSm;
    return PKV_OK;
}

// Timing events: under stream capture they must be recorded as external
// event-record nodes (a plain record would only express a dependency inside
// the graph); outside capture the external flag is not allowed.
cudaError_t record_timing_event(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    if (cs == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    return cudaEventRecord(ev, s);
}

// Validate whole-block copy pairs on the host and launch the copies of
// block_bytes per block in both pools (batches of kCopyPairsPerLaunch).
pkv_status copy_blocks(int NB, const int64_t *pairs, int n, void *k_pool, void *v_pool,
                       size_t block_bytes, cudaStream_t stream) {
    if (n < 0) return fail(PKV_ERR_INVALID_ARG, "num_pairs %d", n);
    if (n == 0) return PKV_OK;
    if (!pairs || !k_pool || !v_pool) return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16))
        return fail(PKV_ERR_INVALID_ARG, "pools must be 16-byte aligned");
    std::unordered_set<int64_t> srcs, dsts;
    for (int i = 0; i < n; ++i) {
        const int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= NB || d < 0 || d >= NB)
            return fail(PKV_ERR_INVALID_ARG, "pair %d (%lld -> %lld) outside [0, %d)", i,
                        (long long)s, (long long)d, NB);
        if (!dsts.insert(d).second)
            return fail(PKV_ERR_INVALID_ARG, "block %lld is the destination of two pairs", (long long)d);
        srcs.insert(s);
    }
    for (int64_t d : dsts)
        if (srcs.count(d))
            return fail(PKV_ERR_INVALID_ARG, "block %lld is both a source and a destination",
                        (long long)d);
    for (int base = 0; base < n; base += pkv::kCopyPairsPerLaunch) {
        pkv::CopyPairs cp;
        const int m = n - base < pkv::kCopyPairsPerLaunch ? n - base : pkv::kCopyPairsPerLaunch;
        for (int i = 0; i < m; ++i) {
            cp.src[i] = pairs[2 * (base + i)];
            cp.dst[i] = pairs[2 * (base + i) + 1];
        }
        cudaError_t e = pkv::launch_block_copy(cp, m, k_pool, v_pool, block_bytes, stream);
        if (e != cudaSuccess) return cuda_fail(e, "block copy launch");
    }
    return PKV_OK;
}

// Test hook state (pkv_debug_set_wait_fault): the wait limit of decode
// launches and how many launches still withhold an arrival.
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<int> g_drop_left{0};

}  // namespace

namespace pkv {
void next_wait_fault(unsigned long long *wait_ns, int *drop_arrival) {
    const unsigned long long w = g_wait_ns.load(std::memory_order_relaxed);
    *wait_ns = w ? w : PKV_WAIT_LIMIT_NS;
    int left = g_drop_left.load(std::memory_order_relaxed);
    *drop_arrival = 0;
    while (left > 0) {
        if (g_drop_left.compare_exchange_weak(left, left - 1, std::memory_order_relaxed)) {
            *drop_arrival = 1;
            break;
        }
    }
}

pkv_status device_error_word(unsigned **out) { return device_error_ptr(out); }

pkv_status set_last_error(pkv_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}
}  // namespace pkv

extern "C" {

const char *pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_OUT_OF_RANGE: return "device-side value out of range";
        case PKV_ERR_TIMEOUT: return "on-chip wait timed out";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_NO_BLOCKS: return "not enough free blocks";
    }
    return "unknown status";
}

const char *pkv_last_error_message(void) { return g_msg; }

pkv_status pkv_debug_set_wait_fault(uint64_t wait_limit_ns, int32_t drop_arrivals) {
    if (drop_arrivals < 0) return fail(PKV_ERR_INVALID_ARG, "drop_arrivals %d", drop_arrivals);
    g_wait_ns.store(wait_limit_ns, std::memory_order_relaxed);
    g_drop_left.store(drop_arrivals, std::memory_order_relaxed);
    return PKV_OK;
}

pkv_status pkv_append(const pkv_cache_desc *cache, const void *k_new, const void *v_new,
                      const int64_t *slot_mapping, int32_t num_tokens, void *k_pool,
                      void *v_pool, void *stream) {
    return pkv_append_ex(cache, k_new, v_new, slot_mapping, num_tokens, k_pool, v_pool, stream,
                         nullptr);
}

pkv_status pkv_append_ex(const pkv_cache_desc *cache, const void *k_new, const void *v_new,
                         const int64_t *slot_mapping, int32_t num_tokens, void *k_pool,
                         void *v_pool, void *stream, const pkv_append_options *options) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_pool || !v_pool)
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(slot_mapping, 8))
        return fail(PKV_ERR_INVALID_ARG, "pointers must be 16-byte aligned (slot_mapping 8)");
    unsigned *err = nullptr;
    if ((st = device_error_ptr(&err)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_append(cache->dtype, k_new, v_new, slot_mapping, num_tokens, k_pool,
                                       v_pool, cache->num_blocks, cache->num_kv_heads,
                                       cache->block_size, cache->head_dim,
                                       options ? (options->inputs_ready != 0) : 0, err,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return PKV_OK;
}

pkv_status pkv_block_copy(const pkv_cache_desc *cache, const int64_t *src_dst_pairs,
                          int32_t num_pairs, void *k_pool, void *v_pool, void *stream) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    const size_t block_bytes = (size_t)cache->num_kv_heads * cache->block_size * cache->head_dim *
                               elem_bytes(cache->dtype);
    return copy_blocks(cache->num_blocks, src_dst_pairs, num_pairs, k_pool, v_pool, block_bytes,
                       static_cast<cudaStream_t>(stream));
}

pkv_status pkv_block_copy_quant(const pkv_qcache_desc *cache, const int64_t *src_dst_pairs,
                                int32_t num_pairs, void *k_codes, void *v_codes, float *k_scales,
                                float *v_scales, void *stream) {
    pkv_status st = check_qcache(cache);
    if (st != PKV_OK) return st;
    if (num_pairs > 0 && (!k_scales || !v_scales))
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (num_pairs > 0 && (!aligned(k_scales, 16) || !aligned(v_scales, 16)))
        return fail(PKV_ERR_INVALID_ARG, "scale pools must be 16-byte aligned");
    const size_t rows = (size_t)cache->num_kv_heads * cache->block_size;
    // pairs are checked by the first call; the second cannot fail on them
    if ((st = copy_blocks(cache->num_blocks, src_dst_pairs, num_pairs, k_codes, v_codes,
                          rows * cache->head_dim, static_cast<cudaStream_t>(stream))) != PKV_OK)
        return st;
    return copy_blocks(cache->num_blocks, src_dst_pairs, num_pairs, k_scales, v_scales,
                       rows * sizeof(float), static_cast<cudaStream_t>(stream));
}

size_t pkv_decode_workspace_bytes_ex(const pkv_cache_desc *cache, int32_t num_q_heads,
                                     int32_t num_ctas) {
    if (check_cache(cache) != PKV_OK) return 0;
    if (num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0 || num_ctas < 0 ||
        num_ctas > PKV_MAX_DECODE_CTAS)
        return 0;
    int C = num_ctas;
    if (C == 0 && max_default_ctas(&C) != PKV_OK) return 0;
    const int G = num_q_heads / cache->num_kv_heads;
    const int GC = G < pkv::kMaxHeadsPerUnit ? G : pkv::kMaxHeadsPerUnit;
    return workspace_for(C, GC, cache->head_dim);
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc *cache, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_context_len) {
    (void)num_seqs;
    (void)max_context_len;
    return pkv_decode_workspace_bytes_ex(cache, num_q_heads, 0);
}

}  // extern "C"

namespace {

// What one decode call reads and writes, whatever the cache format.
struct DecodeArgs {
    int NB, B, Hk, D;
    int q_es;                        // bytes of one q element
    const void *q;
    int S, Hq;
    const void *kp, *vp;
    const float *ks, *vs;            // row scales (8-bit caches) or NULL
    const int32_t *tables;
    int M;
    const int32_t *lens;
    float scale;
    void *out;
    int out_dtype;
    void *ws;
    size_t ws_bytes;
    cudaStream_t stream;
    const pkv_decode_options *opts;
    // fused append (paged caches): each sequence's new row, [S][Hk][D]
    const void *k_new = nullptr, *v_new = nullptr;
    // prefix-aware launch: the work map and the result buffers (one launch)
    const pkv::PrefixMap *pfx_map = nullptr;
    pkv::PrefixBuffers pfx_buf = {nullptr, nullptr, nullptr};
    // flat spans (tables is then NULL): see DecodeParams
    const int32_t *slots = nullptr;
    const int32_t *committed = nullptr;
    size_t slot_stride = 0, v_off = 0;
};

// Host checks shared by the decode entry points (after the cache descriptor).
pkv_status check_decode_args(const DecodeArgs &a) {
    if (a.S < 0) return fail(PKV_ERR_INVALID_ARG, "num_seqs %d", a.S);
    if (!valid_dtype(a.out_dtype)) return fail(PKV_ERR_UNSUPPORTED, "out_dtype %d", a.out_dtype);
    if (a.M < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d", a.M);
    if (!isfinite(a.scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
    return PKV_OK;
}

pkv_status run_decode(const Plan &pl, const DecodeArgs &a) {
    if (a.S == 0) return PKV_OK;
    if (!a.q || !a.kp || !a.vp || (!a.tables && !a.slots) || !a.lens || !a.out)
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(a.q, 16) || !aligned(a.kp, 16) || !aligned(a.vp, 16) ||
        !aligned(a.out, elem_bytes(a.out_dtype)) || !aligned(a.tables, 4) ||
        !aligned(a.slots, 4) || !aligned(a.lens, 4))
        return fail(PKV_ERR_INVALID_ARG, "q and the pools must be 16-byte aligned");
    // flattened tile count must fit in int32
    const int64_t max_tiles_per_unit =
        ((int64_t)a.M * a.B + PKV_TILE_TOKENS - 1) / PKV_TILE_TOKENS;
    const int64_t chunk_seqs = (a.S < pkv::kMaxSeqsPerLaunch ? a.S : pkv::kMaxSeqsPerLaunch) +
                               (a.pfx_map ? a.pfx_map->nv : 0);
    if (chunk_seqs * pl.U * max_tiles_per_unit >= (int64_t)INT32_MAX)
        return fail(PKV_ERR_UNSUPPORTED, "batch x context too large for one launch");

    int C = a.opts ? a.opts->num_ctas : 0;
    pkv_status st;
    if (C < 0 || C > PKV_MAX_DECODE_CTAS)
        return fail(PKV_ERR_INVALID_ARG, "num_ctas %d outside [0, %d]", C, PKV_MAX_DECODE_CTAS);
    if (C == 0 && (st = default_ctas(pl, &C)) != PKV_OK) return st;
    const int pending_tail = a.opts ? a.opts->pending_tail : 0;
    if (pending_tail < 0)
        return fail(PKV_ERR_INVALID_ARG, "pending_tail %d is negative", pending_tail);
    if (pending_tail > 0 && !a.opts->tables_ready)
        return fail(PKV_ERR_INVALID_ARG, "pending_tail needs tables_ready");
    // partial slots: workspace_for counts two per CTA
    const size_t need = workspace_for(C * pl.slots / 2, pl.GC, a.D);
    if (pl.slots > 2 && 2 * C > PKV_MAX_DECODE_CTAS)
        return fail(PKV_ERR_INVALID_ARG, "num_ctas %d above %d for a prefix-aware launch", C,
                    PKV_MAX_DECODE_CTAS / 2);
    if (C > 1 && (!a.ws || a.ws_bytes < need))
        return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    a.ws ? a.ws_bytes : (size_t)0);
    if (a.ws && !aligned(a.ws, 16))
        return fail(PKV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

    unsigned *err = nullptr;
    if ((st = device_error_ptr(&err)) != PKV_OK) return st;

    const int oes = elem_bytes(a.out_dtype);
    cudaEvent_t ev[2] = {nullptr, nullptr};
    if (a.opts)
        for (int i = 0; i < 2; ++i) ev[i] = static_cast<cudaEvent_t>(a.opts->timing_events[i]);

    for (int s0 = 0; s0 < a.S; s0 += pkv::kMaxSeqsPerLaunch) {
        const int S = a.S - s0 < pkv::kMaxSeqsPerLaunch ? a.S - s0 : pkv::kMaxSeqsPerLaunch;
        pkv::DecodeParams p;
        p.q = static_cast<const uint8_t *>(a.q) + (size_t)s0 * a.Hq * a.D * a.q_es;
        p.out = static_cast<uint8_t *>(a.out) + (size_t)s0 * a.Hq * a.D * oes;
        p.out_dtype = a.out_dtype;
        p.block_tables = a.tables ? a.tables + (size_t)s0 * a.M : nullptr;
        p.slots = a.slots ? a.slots + s0 : nullptr;
        p.lse_out = a.opts && a.opts->lse_out ? a.opts->lse_out + (size_t)s0 * a.Hq : nullptr;
        p.committed = a.committed;
        p.slot_stride = a.slot_stride;
        p.v_off = a.v_off;
        p.context_lens = a.lens + s0;
        p.M = a.M;
        p.S = S;
        p.Hq = a.Hq;
        p.Hk = a.Hk;
        p.G = pl.G;
        p.NC = pl.NC;
        p.GC = pl.GC;
        p.U = pl.U;
        p.B = a.B;
        p.NB = a.NB;
        p.scale_log2 = a.scale * 1.4426950408889634f;
        p.ws_cnt = static_cast<unsigned *>(a.ws);
        p.ws_o = a.ws ? reinterpret_cast<float *>(static_cast<uint8_t *>(a.ws) + kCounterBytes)
                      : nullptr;
        p.ws_lse = a.ws ? p.ws_o + (size_t)C * pl.slots * pl.GC * a.D : nullptr;
        p.C = C;
        p.tables_ready = a.opts ? (a.opts->tables_ready != 0) : 0;
        // a later launch of a long batch follows the first one on the stream,
        // not the kernel the caller's promise is about
        p.pending_tail = s0 == 0 ? pending_tail : 0;
        p.err = err;
        p.kp = a.kp;
        p.vp = a.vp;
        p.ks = a.ks;
        p.vs = a.vs;
        pkv::next_wait_fault(&p.wait_ns, &p.drop_arrival);
        p.pb = a.pfx_buf;
        const size_t new_off = (size_t)s0 * a.Hk * a.D * a.q_es;
        p.k_new = a.k_new ? static_cast<const uint8_t *>(a.k_new) + new_off : nullptr;
        p.v_new = a.v_new ? static_cast<const uint8_t *>(a.v_new) + new_off : nullptr;
        const bool first = s0 == 0;
        cudaError_t e;
        if (first && ev[0] && (e = record_timing_event(ev[0], a.stream)) != cudaSuccess)
            return cuda_fail(e, "cudaEventRecord");
        if (a.pfx_map) {
            // one launch for the whole batch (the plan keeps it within one);
            // every read waits for the preceding kernel
            p.pending_tail = 0;
            e = pl.variant->launch_prefix(p, *a.pfx_map, a.stream);
        } else {
            e = pl.variant->launch(p, a.stream);
        }
        if (e != cudaSuccess) return cuda_fail(e, "split-K decode launch");
        if (first && ev[1] && (e = record_timing_event(ev[1], a.stream)) != cudaSuccess)
            return cuda_fail(e, "cudaEventRecord");
    }
    return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_attention_ex(const pkv_cache_desc *cache, const void *q, int32_t num_seqs,
                                   int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, float scale, void *out,
                                   int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                   void *stream, const pkv_decode_options *options) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    DecodeArgs a{cache->num_blocks, cache->block_size, cache->num_kv_heads, cache->head_dim,
                 elem_bytes(cache->dtype), q, num_seqs, num_q_heads, k_pool, v_pool, nullptr,
                 nullptr, block_tables, max_blocks_per_seq, context_lens, scale, out, out_dtype,
                 workspace, workspace_bytes, static_cast<cudaStream_t>(stream), options};
    if ((st = check_decode_args(a)) != PKV_OK) return st;
    Plan pl;
    if ((st = make_plan(cache, num_q_heads, options, &pl)) != PKV_OK) return st;
    return run_decode(pl, a);
}

pkv_status pkv_append_decode_attention(const pkv_cache_desc *cache, const void *q,
                                       int32_t num_seqs, int32_t num_q_heads, const void *k_new,
                                       const void *v_new, void *k_pool, void *v_pool,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, float scale, void *out,
                                       int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                       void *stream, const pkv_decode_options *options) {
    pkv_status st = check_cache(cache);
    if (st != PKV_OK) return st;
    DecodeArgs a{cache->num_blocks, cache->block_size, cache->num_kv_heads, cache->head_dim,
                 elem_bytes(cache->dtype), q, num_seqs, num_q_heads, k_pool, v_pool, nullptr,
                 nullptr, block_tables, max_blocks_per_seq, context_lens, scale, out, out_dtype,
                 workspace, workspace_bytes, static_cast<cudaStream_t>(stream), options};
    if ((st = check_decode_args(a)) != PKV_OK) return st;
    if (num_seqs > 0 && (!k_new || !v_new))
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
        return fail(PKV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    Plan pl;
    if ((st = make_plan(cache, num_q_heads, options, &pl)) != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    // one launch where a fused variant exists (fp16 / bf16 with the tensor-core
    // math); otherwise the append (slots from the tables) and then the decode,
    // which waits for it before it reads the newest rows
    const pkv::DecodeVariant *fv =
        pl.mma ? pkv::find_variant_fused(cache->dtype, cache->head_dim, pl.gmax) : nullptr;
    if (fv) {
        pl.variant = fv;
        a.k_new = k_new;
        a.v_new = v_new;
        return run_decode(pl, a);
    }
    if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out)
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(block_tables, 4) ||
        !aligned(context_lens, 4))
        return fail(PKV_ERR_INVALID_ARG, "q and the pools must be 16-byte aligned");
    unsigned *err = nullptr;
    if ((st = device_error_ptr(&err)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_append(cache->dtype, k_new, v_new, nullptr, num_seqs, k_pool,
                                       v_pool, cache->num_blocks, cache->num_kv_heads,
                                       cache->block_size, cache->head_dim, 0, err,
                                       static_cast<cudaStream_t>(stream), block_tables,
                                       context_lens, max_blocks_per_seq);
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return run_decode(pl, a);
}

pkv_status pkv_decode_attention_quant(const pkv_qcache_desc *cache, const void *q,
                                      int32_t num_seqs, int32_t num_q_heads, const void *k_codes,
                                      const void *v_codes, const float *k_scales,
                                      const float *v_scales, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      float scale, void *out, int32_t out_dtype, void *workspace,
                                      size_t workspace_bytes, void *stream,
                                      const pkv_decode_options *options) {
    pkv_status st = check_qcache(cache);
    if (st != PKV_OK) return st;
    DecodeArgs a{cache->num_blocks, cache->block_size, cache->num_kv_heads, cache->head_dim,
                 elem_bytes(cache->act_dtype), q, num_seqs, num_q_heads, k_codes, v_codes,
                 k_scales, v_scales, block_tables, max_blocks_per_seq, context_lens, scale, out,
                 out_dtype, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), options};
    if ((st = check_decode_args(a)) != PKV_OK) return st;
    Plan pl;
    if ((st = make_plan_quant(cache, num_q_heads, options, &pl)) != PKV_OK) return st;
    if (num_seqs > 0 && (!k_scales || !v_scales))
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(k_scales, 16) || !aligned(v_scales, 16))
        return fail(PKV_ERR_INVALID_ARG, "scale pools must be 16-byte aligned");
    return run_decode(pl, a);
}

pkv_status pkv_append_decode_attention_quant(
    const pkv_qcache_desc *cache, const void *q, int32_t num_seqs, int32_t num_q_heads,
    const void *k_new, const void *v_new, void *k_codes, void *v_codes, float *k_scales,
    float *v_scales, const int32_t *block_tables, int32_t max_blocks_per_seq,
    const int32_t *context_lens, float scale, void *out, int32_t out_dtype, void *workspace,
    size_t workspace_bytes, void *stream, const pkv_decode_options *options) {
    pkv_status st = check_qcache(cache);
    if (st != PKV_OK) return st;
    DecodeArgs a{cache->num_blocks, cache->block_size, cache->num_kv_heads, cache->head_dim,
                 elem_bytes(cache->act_dtype), q, num_seqs, num_q_heads, k_codes, v_codes,
                 k_scales, v_scales, block_tables, max_blocks_per_seq, context_lens, scale, out,
                 out_dtype, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), options};
    if ((st = check_decode_args(a)) != PKV_OK) return st;
    if (num_seqs > 0 && (!k_new || !v_new || !k_scales || !v_scales))
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_scales, 16) ||
        !aligned(v_scales, 16))
        return fail(PKV_ERR_INVALID_ARG, "k_new, v_new and the scale pools must be 16-byte aligned");
    Plan pl;
    if ((st = make_plan_quant(cache, num_q_heads, options, &pl)) != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    // the quantizing append (slots from the tables), then the decode, which
    // waits for it. (A variant of the E4M3 tensor-core decode that quantized
    // each newest row itself, one launch, made the llama-shaped step slower:
    // 66.3 -> 70.2 us.)
    if (!k_codes || !v_codes || !block_tables || !context_lens)
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    unsigned *err = nullptr;
    if ((st = device_error_ptr(&err)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_append_quant(
        cache->code_dtype, cache->act_dtype, k_new, v_new, nullptr, num_seqs, k_codes, v_codes,
        k_scales, v_scales, cache->num_blocks, cache->num_kv_heads, cache->block_size, 0, err,
        static_cast<cudaStream_t>(stream), block_tables, context_lens, max_blocks_per_seq);
    if (e != cudaSuccess) return cuda_fail(e, "quantized append launch");
    return run_decode(pl, a);
}

size_t pkv_decode_quant_workspace_bytes(const pkv_qcache_desc *cache, int32_t num_q_heads,
                                        int32_t num_ctas) {
    if (check_qcache(cache) != PKV_OK) return 0;
    if (num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0 || num_ctas < 0 ||
        num_ctas > PKV_MAX_DECODE_CTAS)
        return 0;
    int C = num_ctas;
    if (C == 0 && max_default_ctas(&C) != PKV_OK) return 0;
    const int G = num_q_heads / cache->num_kv_heads;
    const int GC = G < pkv::kMaxHeadsPerUnit ? G : pkv::kMaxHeadsPerUnit;
    return workspace_for(C, GC, cache->head_dim);
}

pkv_status pkv_append_quant(const pkv_qcache_desc *cache, const void *k_new, const void *v_new,
                            const int64_t *slot_mapping, int32_t num_tokens, void *k_codes,
                            void *v_codes, float *k_scales, float *v_scales, void *stream) {
    return pkv_append_quant_ex(cache, k_new, v_new, slot_mapping, num_tokens, k_codes, v_codes,
                               k_scales, v_scales, stream, nullptr);
}

pkv_status pkv_append_quant_ex(const pkv_qcache_desc *cache, const void *k_new,
                               const void *v_new, const int64_t *slot_mapping,
                               int32_t num_tokens, void *k_codes, void *v_codes,
                               float *k_scales, float *v_scales, void *stream,
                               const pkv_append_options *options) {
    pkv_status st = check_qcache(cache);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_codes || !v_codes || !k_scales || !v_scales)
        return fail(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_codes, 16) ||
        !aligned(v_codes, 16) || !aligned(k_scales, 16) || !aligned(v_scales, 16) ||
        !aligned(slot_mapping, 8))
        return fail(PKV_ERR_INVALID_ARG, "pointers must be 16-byte aligned (slot_mapping 8)");
    unsigned *err = nullptr;
    if ((st = device_error_ptr(&err)) != PKV_OK) return st;
    cudaError_t e = pkv::launch_append_quant(cache->code_dtype, cache->act_dtype, k_new, v_new,
                                             slot_mapping, num_tokens, k_codes, v_codes, k_scales,
                                             v_scales, cache->num_blocks, cache->num_kv_heads,
                                             cache->block_size,
                                             options && options->inputs_ready ? 1 : 0, err,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantized append launch");
    return PKV_OK;
}

pkv_status pkv_decode_attention(const pkv_cache_desc *cache, const void *q, int32_t num_seqs,
                                int32_t num_q_heads, const void *k_pool, const void *v_pool,
                                const int32_t *block_tables, int32_t max_blocks_per_seq,
                                const int32_t *context_lens, float scale, void *out,
                                int32_t out_dtype, void *workspace, size_t workspace_bytes,
                                void *stream) {
    return pkv_decode_attention_ex(cache, q, num_seqs, num_q_heads, k_pool, v_pool, block_tables,
                                   max_blocks_per_seq, context_lens, scale, out, out_dtype,
                                   workspace, workspace_bytes, stream, nullptr);
}

pkv_status pkv_get_error(int32_t *device_error_word, void *stream) {
    if (!device_error_word) return fail(PKV_ERR_INVALID_ARG, "device_error_word is NULL");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned w = 0;
    e = cudaMemcpyFromSymbol(&w, g_pkv_error_word, sizeof(w));
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_pkv_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    *device_error_word = (int32_t)w;
    if (w == 0) return PKV_OK;
    if (w & PKV_DEVERR_TIMEOUT) {
        // a kernel that gave up may have left split-K arrival counters set
        if ((e = pkv::clear_static_scratch(static_cast<cudaStream_t>(stream))) != cudaSuccess)
            return cuda_fail(e, "zeroing the static scratch");
        return fail(PKV_ERR_TIMEOUT, "device error word 0x%x", w);
    }
    return fail(PKV_ERR_OUT_OF_RANGE, "device error word 0x%x", w);
}

}  // extern "C"

// ---------------------------------------------------------------- prefix-aware decode
namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Host plan of one prefix-aware call (include/pkv.h, pkv_decode_attention_prefix).
struct PrefixPlan {
    bool one_launch = false;   // false: the plain decode serves the call
    int G = 0, gmax = 0, per_unit = 0;   // q heads per kv head; variant width; members per prefix unit
    size_t off_res_o = 0, off_res_l = 0, off_fin = 0, bytes = 0;
    pkv::PrefixMap pm;
};

pkv_status plan_prefix(const pkv_cache_desc *c, int32_t S, int32_t Hq, int32_t M,
                       const pkv_prefix_groups *g, const pkv_decode_options *o, PrefixPlan *pp) {
    pkv_status st = check_cache(c);
    if (st != PKV_OK) return st;
    if (!g) return fail(PKV_ERR_INVALID_ARG, "prefix groups are NULL");
    if (S < 0 || M < 1 || Hq < 1 || Hq % c->num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "bad sizes");
    if (g->num_groups < 0 || (S > 0 && !g->group_of_seq) ||
        (g->num_groups > 0 && !g->group_prefix_blocks))
        return fail(PKV_ERR_INVALID_ARG, "bad prefix groups");
    const int32_t num_ctas = o ? o->num_ctas : 0;
    if (num_ctas < 0 || num_ctas > PKV_MAX_DECODE_CTAS)
        return fail(PKV_ERR_INVALID_ARG, "num_ctas %d outside [0, %d]", num_ctas,
                    PKV_MAX_DECODE_CTAS);
    std::vector<std::vector<int32_t>> members(g->num_groups);
    for (int32_t s = 0; s < S; ++s) {
        const int32_t gi = g->group_of_seq[s];
        if (gi < -1 || gi >= g->num_groups)
            return fail(PKV_ERR_INVALID_ARG, "group_of_seq[%d] = %d", s, gi);
        if (gi >= 0) members[gi].push_back(s);
    }
    for (int32_t gi = 0; gi < g->num_groups; ++gi) {
        const int32_t pb = g->group_prefix_blocks[gi];
        if (pb < 1 || pb > M || members[gi].empty())
            return fail(PKV_ERR_INVALID_ARG, "group %d: prefix of %d blocks, %zu members", gi, pb,
                        members[gi].size());
    }
    PrefixPlan &p = *pp;
    const int Hk = c->num_kv_heads, D = c->head_dim;
    p.G = Hq / Hk;
    p.gmax = p.G <= 8 ? 8 : 16;
    p.per_unit = p.gmax / (p.G < 1 ? 1 : p.G);
    int nv = 0;
    for (auto &mem : members) nv += ((int)mem.size() + p.per_unit - 1) / (p.per_unit ? p.per_unit : 1);
    // one launch for 16-bit caches on the tensor cores, kv groups of a whole
    // number of 128-element slice periods (a member's outputs then fall in the
    // same merge slices in a prefix unit as in its own units, and every slice
    // holds part of each) and work lists that fit the map
    p.one_launch = (c->dtype == PKV_F16 || c->dtype == PKV_BF16) && !(o && o->consumer == 1) &&
                   p.G <= 16 && (p.G * D) % 128 == 0 && S + nv <= pkv::kMaxPrefixWork &&
                   g->num_groups > 0;
    int C = num_ctas;
    if (C == 0 && (st = max_default_ctas(&C)) != PKV_OK) return st;
    if (!p.one_launch) {
        p.bytes = workspace_for(C, p.G < pkv::kMaxHeadsPerUnit ? p.G : pkv::kMaxHeadsPerUnit, D);
        return PKV_OK;
    }
    // the work map: the groups' prefix units (per_unit members each), then every sequence
    pkv::PrefixMap &m = p.pm;
    m.nv = nv;
    int w = 0, k = 0;
    for (int32_t gi = 0; gi < g->num_groups; ++gi) {
        const int m_first = k;
        for (int32_t s : members[gi]) m.members[k++] = (int16_t)s;
        for (int j = 0; j < (int)members[gi].size(); j += p.per_unit) {
            const int n = (int)members[gi].size() - j < p.per_unit ? (int)members[gi].size() - j
                                                                  : p.per_unit;
            m.w[w++] = pkv::PrefixWork{g->group_prefix_blocks[gi], members[gi][0], m_first + j, n};
        }
    }
    for (int32_t s = 0; s < S; ++s) {
        const int32_t gi = g->group_of_seq[s];
        m.w[nv + s] = pkv::PrefixWork{gi >= 0 ? g->group_prefix_blocks[gi] : 0, s, 0, 0};
    }
    // workspace: the split-K part (units carry up to gmax heads), then the
    // prefix and suffix result rows, then the (sequence, kv head) counters
    // four partial slots per CTA (two sections), arrival counters for 2 C
    if (2 * C > PKV_MAX_DECODE_CTAS)
        return fail(PKV_ERR_INVALID_ARG, "num_ctas %d above %d for a prefix-aware launch", C,
                    PKV_MAX_DECODE_CTAS / 2);
    p.off_res_o = align256(workspace_for(2 * C, p.per_unit * p.G, D));
    p.off_res_l = p.off_res_o + align256((size_t)2 * S * Hq * D * sizeof(float));
    p.off_fin = p.off_res_l + align256((size_t)2 * S * Hq * pkv::kMergeSlices * sizeof(float));
    p.bytes = p.off_fin + align256((size_t)S * Hk * pkv::kMergeSlices * sizeof(unsigned));
    return PKV_OK;
}

}  // namespace

extern "C" {

size_t pkv_decode_prefix_workspace_bytes(const pkv_cache_desc *cache, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_blocks_per_seq,
                                         const pkv_prefix_groups *groups, int32_t num_ctas) {
    pkv_decode_options o = {};
    o.num_ctas = num_ctas;
    std::unique_ptr<PrefixPlan> pp(new PrefixPlan());
    if (plan_prefix(cache, num_seqs, num_q_heads, max_blocks_per_seq, groups, &o, pp.get()) !=
        PKV_OK)
        return 0;
    return pp->bytes;
}

pkv_status pkv_decode_attention_prefix(const pkv_cache_desc *cache, const void *q,
                                       int32_t num_seqs, int32_t num_q_heads, const void *k_pool,
                                       const void *v_pool, const int32_t *block_tables,
                                       int32_t max_blocks_per_seq, const int32_t *context_lens,
                                       float scale, const pkv_prefix_groups *groups, void *out,
                                       int32_t out_dtype, void *workspace,
                                       size_t workspace_bytes, void *stream,
                                       const pkv_decode_options *options) {
    std::unique_ptr<PrefixPlan> pp(new PrefixPlan());
    pkv_status st = plan_prefix(cache, num_seqs, num_q_heads, max_blocks_per_seq, groups,
                                options, pp.get());
    if (st != PKV_OK) return st;
    if (!pp->one_launch)
        return pkv_decode_attention_ex(cache, q, num_seqs, num_q_heads, k_pool, v_pool,
                                       block_tables, max_blocks_per_seq, context_lens, scale, out,
                                       out_dtype, workspace, workspace_bytes, stream, options);
    DecodeArgs a{cache->num_blocks, cache->block_size, cache->num_kv_heads, cache->head_dim,
                 elem_bytes(cache->dtype), q, num_seqs, num_q_heads, k_pool, v_pool, nullptr,
                 nullptr, block_tables, max_blocks_per_seq, context_lens, scale, out, out_dtype,
                 workspace, workspace_bytes, static_cast<cudaStream_t>(stream), options};
    if ((st = check_decode_args(a)) != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    if (!workspace || workspace_bytes < pp->bytes)
        return fail(PKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", pp->bytes,
                    workspace ? workspace_bytes : (size_t)0);
    Plan pl;
    pl.G = pp->G;
    pl.GC = pp->per_unit * pp->G;   // heads a unit may carry: the workspace's partial rows
    pl.NC = 1;
    pl.U = cache->num_kv_heads;
    pl.mma = true;
    pl.gmax = pp->gmax;
    pl.slots = 4;
    pl.variant = pkv::find_variant_prefix(cache->dtype, cache->head_dim, pp->gmax);
    if (!pl.variant) return fail(PKV_ERR_UNSUPPORTED, "no kernel variant for this shape");
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.pfx_map = &pp->pm;
    a.pfx_buf = pkv::PrefixBuffers{reinterpret_cast<float *>(ws + pp->off_res_o),
                                   reinterpret_cast<float *>(ws + pp->off_res_l),
                                   reinterpret_cast<unsigned *>(ws + pp->off_fin)};
    return run_decode(pl, a);
}

}  // extern "C"

// ---------------------------------------------------------------- flat spans
namespace pkv {

pkv_status decode_flat(const FlatGeom &g, const void *q, int32_t S, int32_t Hq,
                       const int32_t *slots, const int32_t *lens, float scale, void *out,
                       int32_t out_dtype, void *ws, size_t ws_bytes, cudaStream_t stream,
                       const pkv_decode_options *o) {
    if (o && o->consumer == 1)
        return fail(PKV_ERR_UNSUPPORTED, "flat spans use the tensor-core math (consumer 1 given)");
    DecodeArgs a{g.num_slots, kFlatRowsPerGroup, g.Hk, g.D, elem_bytes(g.dtype), q, S, Hq,
                 g.k_base, g.k_base, nullptr, nullptr, nullptr,
                 g.capacity / kFlatRowsPerGroup, lens, scale, out, out_dtype, ws, ws_bytes,
                 stream, o};
    a.slots = slots;
    a.committed = g.committed;
    a.slot_stride = g.slot_stride;
    a.v_off = g.v_off;
    pkv_status st = check_decode_args(a);
    if (st != PKV_OK) return st;
    Plan pl;
    if ((st = plan_groups(g.Hk, Hq, o, true, &pl)) != PKV_OK) return st;
    pl.variant = find_variant_flat(g.dtype, g.D, pl.gmax);
    if (!pl.variant) return fail(PKV_ERR_UNSUPPORTED, "no kernel variant for this shape");
    return run_decode(pl, a);
}

size_t flat_workspace_bytes(const FlatGeom &g, int32_t Hq, int32_t num_ctas) {
    if (Hq < 1 || Hq % g.Hk != 0 || num_ctas < 0 || num_ctas > PKV_MAX_DECODE_CTAS) return 0;
    int C = num_ctas;
    if (C == 0 && max_default_ctas(&C) != PKV_OK) return 0;
    const int G = Hq / g.Hk;
    return workspace_for(C, G < kMaxHeadsPerUnit ? G : kMaxHeadsPerUnit, g.D);
}

}  // namespace pkv
