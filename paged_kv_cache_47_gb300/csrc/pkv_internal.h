// Internal declarations shared by libpkv's translation units (not part of the
// C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

// Default limit of every on-chip wait of a decode launch.
#define PKV_WAIT_LIMIT_NS 2000000000ull  // 2 s: far above any legitimate wait

namespace pkv {

constexpr int kConsumerWarps = 4;                  // math warps of the split-K kernel
constexpr int kMergeSlices = 4;                    // workspace slices of a cut unit's partial
constexpr int kProducerWarps = 4;                  // gather (cp.async) warps
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kMaxSeqsPerLaunch = 1024;            // larger batches are launched in chunks
constexpr int kMaxCtasPerSm = 2;                   // cap used to size the workspace
constexpr int kMaxHeadsPerUnit = 16;               // q heads carried by one work unit

// Per-tile record the producer warp hands to the math warps with each stage.
struct TileMeta {
    int s;       // sequence (within this launch)
    int h0;      // first q head of the unit
    int gca;     // q heads in the unit
    int ntok;    // valid tokens in this tile (1..64)
    int flags;   // kFirst | kLast | kWhole
    int slot;    // partial slot (0/1) when the segment is not a whole unit
    int tu;      // first tile of the unit (flattened tile index of the launch)
    int nu;      // tiles of the unit
};
constexpr int kFirst = 1;  // first tile of this CTA's segment of a unit
constexpr int kLast = 2;   // last tile of this CTA's segment of a unit
constexpr int kWhole = 4;  // the segment is the whole unit: write the output directly
constexpr int kNewRow = 8; // fused append: the tile's last row is the context's newest,
                           // whose K/V rows wait in the stage's side slot

// ---------------------------------------------------------------- prefix-aware decode
// One launch decodes sequences that share leading blocks: each group's shared
// prefix is a run of "virtual" work sequences placed first in the work list,
// each carrying up to GMAX / G members' q heads under every kv head; each
// grouped sequence's own units cover its context past the prefix. A unit's
// result for a member goes to a workspace row (prefix or suffix); per
// (sequence, kv head, merge slice) an arrival counter takes one count when
// the slice of the prefix result is written and one for the suffix result's,
// and the warp that brings it to two merges that slice of the two by
// log-sum-exp into `out`. A member
// whose context ends with the prefix gets its prefix result directly.
constexpr int kMaxPrefixWork = 1024;   // virtual + real work sequences of one launch
struct PrefixWork {
    int32_t blocks;   // shared prefix blocks (virtual: the prefix; real: its group's, 0 = none)
    int32_t row;      // table row the work sequence reads (virtual: a member; real: itself)
    int32_t m0, nm;   // virtual: first member in members[], member count; real: 0, 0
};
struct PrefixMap {
    int32_t nv;                               // virtual work sequences (first in the list)
    PrefixWork w[kMaxPrefixWork];             // [nv + S]
    int16_t members[kMaxPrefixWork];          // sequence ids, each group's together
};
struct NoPrefixMap {};
// Workspace pointers of the prefix-aware launch (NULL otherwise).
struct PrefixBuffers {
    float *res_o;      // [2][S][Hq][D]: prefix, then suffix result rows
    float *res_l;      // [2][S][Hq][kMergeSlices]: their log2-sum-exp2, a copy per slice
    unsigned *fin;     // [S][Hk][kMergeSlices] arrival counters, zero between calls
};

struct DecodeParams {
    const void *q;              // [S][Hq][D]
    void *out;                  // [S][Hq][D] in out_dtype
    int out_dtype;
    const int32_t *block_tables;  // [S][M]
    const int32_t *context_lens;  // [S]
    int M;                      // table width
    int S, Hq, Hk, G;           // sequences, q heads, kv heads, group size
    int NC, GC, U;              // head chunks per kv head, heads per chunk, units per seq
    int B, NB;                  // block size, physical blocks
    float scale_log2;           // scale * log2(e)
    // Split-K workspace. A unit cut by CTA boundaries is indexed by its first
    // owner c_first (a CTA starts at most one unit that runs past its range).
    // Math warp w < kMergeSlices of each CTA holding a partial owns a fixed
    // slice of the unit's (head, d) elements: it writes that slice, then
    // counts itself in ws_cnt[c_first][w]; the warp that arrives last merges
    // the slice over all partials and puts the counter back to zero.
    unsigned *ws_cnt;           // [C][kMergeSlices] arrival counters, zero between calls
    float *ws_o;                // [C][2][GC][D] partial outputs (normalised)
    float *ws_lse;              // [C][2][kMergeSlices][GC] partial log2-sum-exp2, one
                                //                copy per owning warp
    int C;                      // CTAs of the split-K launch
    int tables_ready;           // lengths / tables / slots may be read before the
                                // preceding kernel on the stream finishes
    int pending_tail;           // > 0: q and the rows below L - pending_tail may be
                                // read before it finishes too (the last
                                // pending_tail rows of a sequence and every
                                // store wait for it)
    unsigned *err;              // device error word
    const void *kp, *vp;        // pools [NB][Hk][B][D] (elements, or 8-bit codes)
    const float *ks, *vs;       // 8-bit caches: row scales [NB][Hk][B]; else unused
    // Flat spans (decode over one contiguous span per sequence instead of
    // blocks): kp is K of slot 0, slot i starts slot_stride bytes further, V
    // sits v_off bytes after K, and token t of kv head g is row t * Hk + g.
    // NB is then the number of slots and M * B the span capacity in tokens.
    float *lse_out;             // optional [S][Hq]: log2 sum_t exp(scaled score)
    const int32_t *slots;       // [S] batch entry -> slot (flat spans only)
    const int32_t *committed;   // [NB] tokens of each slot backed by memory
    size_t slot_stride, v_off;
    // Append fused into the decode (paged 16/32-bit caches; NULL = none):
    // k_new / v_new [S][Hk][D] hold the row each sequence adds at position
    // L - 1. The attention takes that row from here instead of the pool, and
    // the producer warps write it into its slot (the block table's entry for
    // position L - 1) once they have issued their last tile.
    const void *k_new, *v_new;
    // Bounded waits: every mbarrier wait of the launch gives up after wait_ns
    // (PKV_WAIT_LIMIT_NS by default). drop_arrival != 0 is a test hook: the
    // first producer thread of CTA 0 withholds its arrival on its first stage.
    unsigned long long wait_ns;
    int drop_arrival;
    PrefixBuffers pb;           // prefix-aware launch only
};

// Wait limit and withheld arrivals for the next decode launches (test hook,
// pkv_debug_set_wait_fault); returns the limit and whether this launch drops.
void next_wait_fault(unsigned long long *wait_ns, int *drop_arrival);

using SplitLaunchFn = cudaError_t (*)(const DecodeParams &, cudaStream_t);
using PrefixLaunchFn = cudaError_t (*)(const DecodeParams &, const PrefixMap &, cudaStream_t);
using MaxCtasFn = int (*)();

struct DecodeVariant {
    SplitLaunchFn launch;       // NULL for prefix-aware variants
    MaxCtasFn max_ctas_per_sm;  // occupancy of the split-K kernel (0 = cannot run)
    PrefixLaunchFn launch_prefix = nullptr;   // prefix-aware variants only
};

// Variant lookup per K/V dtype (defined in decode_<dtype>.cu). gmax is the
// compile-time head capacity (1, 2, 4, 8 or 16); mma selects the tensor-core
// math (16-bit dtypes, gmax 8 or 16). Returns nullptr if not built.
const DecodeVariant *find_variant_f32(int D, int gmax, bool mma);
const DecodeVariant *find_variant_f16(int D, int gmax, bool mma);
const DecodeVariant *find_variant_bf16(int D, int gmax, bool mma);
// Variants with the append fused in (decode_fused.cu): fp16 / bf16, tensor-
// core math, D 64 or 128, gmax 8 or 16; nullptr for any other shape.
const DecodeVariant *find_variant_fused(int dtype, int D, int gmax);
// Prefix-aware variants (decode_prefix.cu): fp16 / bf16, tensor-core math, D 64
// or 128, gmax 8 or 16.
const DecodeVariant *find_variant_prefix(int dtype, int D, int gmax);
// 8-bit caches (decode_quant.cu): code_dtype PKV_INT8 / PKV_FP8_E4M3, q in
// act_dtype PKV_F16 / PKV_BF16, tensor-core math, D = 128, gmax 8 or 16.
const DecodeVariant *find_variant_quant(int code_dtype, int act_dtype, int D, int gmax);
// Flat spans (decode_flat.cu): fp16 / bf16, tensor-core math, D 64 or 128, gmax 8 or 16.
const DecodeVariant *find_variant_flat(int dtype, int D, int gmax);

// Flat spans (flat_cache.cu owns the memory; pkv_api.cu runs the decode).
// The split kernel's producer splits a tile's rows into groups as it splits
// them into pool blocks; flat spans use groups of this many rows.
constexpr int kFlatRowsPerGroup = 16;
struct FlatGeom {
    const void *k_base;          // K span of slot 0
    size_t slot_stride, v_off;   // bytes
    const int32_t *committed;    // device [num_slots]
    int32_t num_slots, capacity, Hk, D, dtype;
};
pkv_status decode_flat(const FlatGeom &g, const void *q, int32_t S, int32_t Hq,
                       const int32_t *slots, const int32_t *lens, float scale, void *out,
                       int32_t out_dtype, void *ws, size_t ws_bytes, cudaStream_t stream,
                       const pkv_decode_options *o);
size_t flat_workspace_bytes(const FlatGeom &g, int32_t Hq, int32_t num_ctas);

// The device error word of the current device (PKV_DEVERR_* bits).
pkv_status device_error_word(unsigned **out);

// Zero pkv_decode_attention_static's scratch on the current device (after a
// timed-out wait may have left arrival counters set): ordered on `stream` and
// complete when it returns.
cudaError_t clear_static_scratch(cudaStream_t stream);

// Record the text pkv_last_error_message returns on this thread; returns st.
pkv_status set_last_error(pkv_status st, const char *fmt, ...);

// slot_mapping NULL: token i is the newest of sequence i and goes to the
// block table's slot of position context_lens[i] - 1 (tables [num_tokens][M]).
cudaError_t launch_append(int dtype, const void *k_new, const void *v_new,
                          const int64_t *slot_mapping, int num_tokens, void *k_pool, void *v_pool,
                          int NB, int Hk, int B, int D, int inputs_ready, unsigned *err,
                          cudaStream_t st, const int32_t *tables = nullptr,
                          const int32_t *lens = nullptr, int M = 0);

// 8-bit caches (append_quant.cu): D = 128.
// slots NULL: token i is sequence i and its slot is position lens[i] - 1 of
// its table row (tables [num_tokens][M])
cudaError_t launch_append_quant(int code_dtype, int act_dtype, const void *k_new,
                                const void *v_new, const int64_t *slots, int num_tokens,
                                void *k_codes, void *v_codes, float *k_scales, float *v_scales,
                                int NB, int Hk, int B, int inputs_ready, unsigned *err,
                                cudaStream_t st, const int32_t *tables = nullptr,
                                const int32_t *lens = nullptr, int M = 0);

constexpr int kCopyPairsPerLaunch = 128;
struct CopyPairs {
    long long src[kCopyPairsPerLaunch];
    long long dst[kCopyPairsPerLaunch];
};
cudaError_t launch_block_copy(const CopyPairs &pairs, int n, void *k_pool, void *v_pool,
                              size_t block_bytes, cudaStream_t st);

}  // namespace pkv
