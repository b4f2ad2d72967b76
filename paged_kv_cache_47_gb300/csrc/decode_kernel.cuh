// Split-K paged decode attention for sm_103a.
//
// What it computes ("PagedAttention — Math + Memory Model", section
// "PagedAttention: blocks and the block table"; "KV-cache paging in vLLM",
// section "The Attention Kernel Change"): for every sequence and q head,
// softmax(scale * q K^T) V over the sequence's context, where the K/V rows of
// token t live at offset t % B of physical block block_tables[s][t / B].
//
// How (GB300 design):
//  * Persistent, stream-K: one CTA per SM (x occupancy) takes an equal share
//    of the flattened (sequence, kv-head unit, tile) space (decomp.h); tiles
//    are 64 tokens, 128 for the 8-bit variants with one mma n-tile. Whole units are written directly. A unit cut by CTA
//    boundaries leaves one partial per CTA; after its last tile each math
//    warp counts its slices of those partials in per-unit arrival counters,
//    and the warp that completes a count merges that slice by log-sum-exp
//    (merge_slice). No CTA ever waits for another.
//  * The last four warps are producers: they walk the CTA's tiles, read block-table
//    entries a few tiles ahead, and gather each (physical block, kv head)
//    chunk with 16-byte cp.async copies into a ring of NST shared-memory
//    stages, written in the 128-byte-swizzled order the math warps read
//    without bank conflicts. Completion is tracked by mbarriers
//    (cp.async.mbarrier.arrive). The copy engine (TMA) is not used for K/V:
//    on GB300 it sustains only about six requests per microsecond per SM, so
//    with the 2-8 KB chunks of a paged cache it reaches 2.2-5.5 TB/s, while
//    16-byte loads reach 6.2-6.6 TB/s on the same random-chunk pattern.
//    The unit's q rows ride along with its first tile.
//  * The first CW warps (4, or 8 on 128-token tiles) do the math: each takes
//    16 of the tile's tokens and keeps its own online-softmax state (running
//    max m, sum l, accumulator) in fp32 registers, in base 2 with
//    scale*log2(e) folded in. At the end of a segment they combine their
//    states through shared memory.
//  * Math: on 16-bit data the products run on tensor cores (mma.sync
//    m16n8k16, tokens as M, q heads as N padded to 8, fp32 accumulate; P is
//    split into hi+lo 16-bit parts so the PV product keeps fp32-level
//    accuracy). 8-bit codes go from shared memory straight into the mma
//    fragments as exact fp16 values. On fp32 data (or when forced) they run
//    on CUDA cores with each lane owning a slice of head_dim (reduce-scatter
//    for the dot products).
//  * Every mbarrier wait is bounded (device_utils.cuh); there is no
//    __syncthreads or named barrier after the producer/consumer split.
#pragma once

#include <cuda_fp8.h>
#include <math_constants.h>

#include <atomic>
#include <type_traits>

#include "decomp.h"
#include "device_utils.cuh"
#include "pkv_internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// compile-time shared-memory plan of one kernel variant
// ---------------------------------------------------------------------------
// T is the activation type (q, k_new / v_new); QK selects the cache format:
// 0 = T elements, kQuantInt8 / kQuantE4m3 = 8-bit codes with one fp32 scale
// per (token, kv head) row.
constexpr int kQuantInt8 = 1;
constexpr int kQuantE4m3 = 2;

// 8-bit variants with one mma n-tile take 128-token tiles and eight math
// warps: an 8-bit tile carries half the bytes of a 16-bit one, so twice the
// tokens keep the producer's per-tile cost and the math warps' per-tile
// latency below the time HBM takes to deliver it. Every other variant takes
// 64-token tiles and four math warps.
constexpr bool big_tiles(int QK, int GMAX) { return QK != 0 && GMAX <= 8; }
constexpr int tile_tokens(int QK, int GMAX) { return big_tiles(QK, GMAX) ? 128 : PKV_TILE_TOKENS; }
// E4M3 caches with one mma n-tile run both products on the 5th-generation
// tensor cores (tcgen05.mma kind::f8f6f4, accumulators in tensor memory):
// the codes are mma operands as they are, so no math warp converts them.
// Their math warps form kTcGroups groups of four that take turns on tiles.
// Units of up to 4 q heads take a 4-head variant (less code per tile).
constexpr bool tc_path(int QK, int GMAX) { return QK == kQuantE4m3 && (GMAX == 4 || GMAX == 8); }
constexpr int kTcGroups = 3;
constexpr int math_warps(int QK, int GMAX) {
    return tc_path(QK, GMAX) ? 4 * kTcGroups : big_tiles(QK, GMAX) ? 8 : kConsumerWarps;
}
constexpr int kernel_threads(int QK, int GMAX) { return 32 * (math_warps(QK, GMAX) + kProducerWarps); }
// 16-bit tensor-core variants of up to 8 heads a unit run two CTAs per SM
// (a two-stage ring each, at most 128 registers a thread): one CTA's prologue
// and merge tail overlap the other's steady state, and with programmatic
// launch the next kernel's CTAs start beside this one's. Measured on the
// same box, 1 -> 2 CTAs per SM: llama-shaped step 103.4 -> 102.1 us, OPT-13B
// decode 924 -> 881 us, long context B = 32 458 -> 425 us, shared prefix with
// short suffixes 57.6 -> 47.8 us. The prefix-aware variants stay at one
// (274 -> 452 us with two).
constexpr bool two_ctas(int QK, int GMAX, bool MMA, bool PFX) {
    return QK == 0 && MMA && GMAX == 8 && !PFX;
}

// Pending final arrivals a merge-slice warp can hold (prefix-aware variants).
constexpr int kFinCap = 32;

template <typename T, int D, int GMAX, bool MMA, int QK = 0, bool FUSED = false, bool PFX = false>
struct SplitCfg {
    static constexpr int ES = QK ? 1 : (int)sizeof(T);  // bytes of one cache element
    static constexpr int ROWB = D * ES;              // bytes of one K or V row
    static constexpr int QROWB = D * (int)sizeof(T); // bytes of one q row
    static constexpr int NP = ROWB / 128;            // 128-byte swizzle planes per row
    static constexpr int TT = tile_tokens(QK, GMAX);   // tokens per tile
    static constexpr int CW = math_warps(QK, GMAX);    // math warps
    static constexpr int THREADS = kernel_threads(QK, GMAX);
    static constexpr int PLANE = TT * 128;
    static constexpr int KVB = NP * PLANE;           // bytes of one tile of K (or V)
    static constexpr int SCB = QK ? 1024 : 0;        // K then V scales of the tile (2 x 256 B)
    static constexpr int QB = ((GMAX * QROWB + 1023) / 1024) * 1024;
    // fused append: the newest row's K then V (side slot, 1 KB-aligned)
    static constexpr int NEWB = FUSED ? ((2 * ROWB + 1023) / 1024) * 1024 : 0;
    static constexpr int STAGE = 2 * KVB + SCB + QB + NEWB; // multiple of 1024
    static constexpr int NTN = GMAX / 8;             // mma n-tiles (MMA only)
    static constexpr bool TC = tc_path(QK, GMAX);
    static constexpr int NG = TC ? CW / 4 : 0;        // warp groups (TC)
    // combine entries of the output: one per math warp, one per warp group (TC)
    static constexpr int CWC = TC ? NG : CW;
    static constexpr int COMB_O = CWC * GMAX * D * 4;
    static constexpr int COMB_ML = 2 * CW * GMAX * 4;
    static constexpr int PBUF = (MMA && !TC) ? CW * NTN * 2 * 256 : 0;
    // TC: per warp group, the q parts and the p parts (mma B operands,
    // 1024-byte aligned; 2 KB each for units of up to 4 heads, 4 KB for 8);
    // then the max-exchange slots, q scales, the tensor-memory address and the
    // group barriers
    static constexpr int TCG = GMAX <= 4 ? 4096 : 8192;   // bytes per group
    static constexpr int TCB = TC ? NG * TCG : 0;
    // exchange slots (per group 2 slots x 4 warps x XS bytes: GMAX maxima and
    // the V scale maximum), q scales (per group 8 floats), the TMEM address,
    // then 4 NG + 2 barriers (8-byte aligned); the region starts 16-byte aligned
    static constexpr int XS = GMAX <= 4 ? 32 : 64;
    static_assert(!TC || 4 * (GMAX + 1) <= XS, "exchange slot too small");
    static constexpr int TCX_QSC = NG * 8 * XS;
    static constexpr int TCX_TSLOT = TCX_QSC + NG * 32;
    static constexpr int TCX_BAR = TCX_TSLOT + 16;
    static constexpr int TCX = TC ? ((TCX_BAR + (4 * NG + 2) * 8 + 16 + 255) / 256) * 256 : 0;
    static constexpr int TMEM_COLS = NG <= 2 ? 128 : NG <= 4 ? 256 : 512;   // S, O: 64 columns per group
    // work sequences: tile prefix and length (and, prefix-aware, the table offset)
    static constexpr int SEQ_MAX = (2 * kMaxSeqsPerLaunch + 1) * 4 + (PFX ? kMaxPrefixWork * 6 : 0);
    static constexpr int FINB = PFX ? kMergeSlices * kFinCap * 4 : 0;
    static constexpr int SMEM_LIMIT = two_ctas(QK, GMAX, MMA, PFX) ? 112 * 1024 : 227 * 1024;
    static constexpr int PER_STAGE_EXTRA = (int)sizeof(TileMeta) + 16;  // meta + 2 barriers
    static constexpr int FIXED = 1024 /*alignment slack*/ + COMB_O + COMB_ML + PBUF + FINB +
                                 TCB + TCX + 16 /*comb bars*/ + SEQ_MAX + 64;
    static constexpr int NST_FIT = (SMEM_LIMIT - FIXED) / (STAGE + PER_STAGE_EXTRA);
    static constexpr int NST = NST_FIT > 8 ? 8 : NST_FIT;
    static_assert(NST >= 2, "shared-memory plan leaves fewer than two stages");
    static_assert(ROWB % 128 == 0, "rows must be whole 128-byte planes");
    static_assert(!QK || MMA, "8-bit caches use the tensor-core math");

    // offsets from the 1024-aligned base
    static constexpr int OFF_TC = NST * STAGE;
    static constexpr int OFF_META = OFF_TC + TCB;
    static constexpr int OFF_FULL = OFF_META + NST * (int)sizeof(TileMeta);
    static constexpr int OFF_EMPTY = OFF_FULL + NST * 8;
    static constexpr int OFF_CBAR = OFF_EMPTY + NST * 8;   // comb_full, comb_empty
    static constexpr int OFF_COMB_O = OFF_CBAR + 16;
    static constexpr int OFF_COMB_M = OFF_COMB_O + COMB_O;
    static constexpr int OFF_COMB_L = OFF_COMB_M + CW * GMAX * 4;
    static constexpr int OFF_PBUF = OFF_COMB_L + CW * GMAX * 4;
    static constexpr int OFF_FIN = OFF_PBUF + PBUF;
    static constexpr int OFF_TCX = OFF_FIN + FINB;
    static constexpr int OFF_SEQ = OFF_TCX + TCX;

    // W work sequences (the batch, plus the virtual prefix ones when prefix-aware,
    // with their table offsets and the member list)
    static size_t smem_bytes(int W) {
        return 1024 + OFF_SEQ + (size_t)(2 * W + 1) * 4 + (PFX ? (size_t)W * 6 + 4 : 0);
    }
};

// ---------------------------------------------------------------------------
// per-sequence tile prefix
// ---------------------------------------------------------------------------
// seq_len[s]   = context length clamped to [0, M*B] (a clamp flags the error word)
// seq_prefix[s]= U * sum_{s'<s} ceil(seq_len[s'] / 64), seq_prefix[S] = NT
// Prefix-aware launches (PFX): W = nv + S work sequences; virtual w < nv spans
// its group's prefix, real w = nv + s the context of s past its group's
// prefix (a context shorter than the prefix flags the error word and counts
// 0); seq_tab[w] is the offset of the work sequence's first table entry.
// members[] (the sequence ids of the prefix units) is copied to shared memory.
// Ends with __syncthreads(); all threads of the block must call it.
template <bool FLAT, int TT, bool PFX = false, typename PM = NoPrefixMap>
__device__ __forceinline__ void build_seq_arrays(const DecodeParams &p, int W, int *seq_prefix,
                                                 int *seq_len, bool report, const PM &pm = PM{},
                                                 int *seq_tab = nullptr,
                                                 int16_t *members = nullptr) {
    const int tid = threadIdx.x;
    const int max_len = p.M * p.B;
    if constexpr (PFX)
        for (int i = tid; i < p.S; i += blockDim.x) members[i] = pm.members[i];
    for (int s = tid; s < W; s += blockDim.x) {
        int bad = 0;
        int L;
        if constexpr (FLAT) {
            // a flat span holds at most the tokens its slot has memory for
            const int slot = p.slots[s];
            if (slot < 0 || slot >= p.NB) {
                if (report) atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
                L = 0;
            } else {
                L = pkv_clamp_len(p.context_lens[s], min(max_len, p.committed[slot]), &bad);
            }
        } else if constexpr (PFX) {
            const PrefixWork wk = pm.w[s];
            if (s < pm.nv) {
                L = wk.blocks * p.B;
            } else {
                const int Lc = pkv_clamp_len(p.context_lens[s - pm.nv], max_len, &bad);
                const int sh = wk.blocks * p.B;
                if (Lc < sh) bad = 1;
                L = Lc < sh ? 0 : Lc - sh;
            }
            seq_tab[s] = wk.row * p.M + (s < pm.nv ? 0 : wk.blocks);
        } else {
            L = pkv_clamp_len(p.context_lens[s], max_len, &bad);
        }
        if (bad && report) atomicOr(p.err, PKV_DEVERR_CONTEXT);
        seq_len[s] = L;
    }
    __syncthreads();
    if (tid < 32) {
        const int lane = tid;
        int running = 0;
        for (int base = 0; base < W; base += 32) {
            const int s = base + lane;
            const int n = (s < W) ? pkv_tiles_of_len(seq_len[s], TT) * p.U : 0;
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (s < W) seq_prefix[s] = running + incl - n;
            running += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) seq_prefix[W] = running;
    }
    __syncthreads();
}

// Swizzled shared-memory address of 16-byte chunk `chunk` (0..8*NP-1) of row r
// in a tile stored as NP planes of [64 rows][128 bytes] with a 128-byte
// XOR swizzle (chunk index XOR row%8 within each 1024-byte atom).
template <int TT = PKV_TILE_TOKENS>
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int chunk) {
    const int pl = chunk >> 3, c = chunk & 7;
    return base + pl * (TT * 128) + r * 128 + ((c ^ (r & 7)) << 4);
}

// ---------------------------------------------------------------------------
// small vector loads from shared memory
// ---------------------------------------------------------------------------
template <typename T, int N>
__device__ __forceinline__ void lds_vec(uint32_t addr, float (&out)[N]) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (N == 4) {
            float4 v;
            asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                         : "r"(addr));
            out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
        } else {
            static_assert(N == 2, "");
            float2 v;
            asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
            out[0] = v.x; out[1] = v.y;
        }
    } else {
        uint32_t w[N / 2];
        if constexpr (N == 4) {
            asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(addr));
        } else {
            static_assert(N == 2, "");
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[0]) : "r"(addr));
        }
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const T *h = reinterpret_cast<const T *>(&w[i]);
            out[2 * i] = Elem<T>::to_f32(h[0]);
            out[2 * i + 1] = Elem<T>::to_f32(h[1]);
        }
    }
}

// ---------------------------------------------------------------------------
// 8-bit codes -> fp16 (exact: every int8 and E4M3 value is an fp16 value)
// ---------------------------------------------------------------------------
// Four codes (lowest address in the low byte) -> two fp16 pairs.
// The bias int8 codes carry into the fp16 mma operands.
constexpr float kInt8Bias = 1152.f;

template <int QK>
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    if constexpr (QK == kQuantInt8) {
        // byte b + 128 placed under the fp16 exponent of 1024 (0x64nn) reads
        // as b + 1152 exactly; the products keep that bias, and the scores and
        // outputs take it off (kInt8Bias times the sum of q, resp. of p)
        const uint32_t u = w ^ 0x80808080u;
        asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
        asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
    } else {
        const __half2_raw a = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
        const __half2_raw b = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
        lo = (uint32_t)a.x | ((uint32_t)a.y << 16);
        hi = (uint32_t)b.x | ((uint32_t)b.y << 16);
    }
}

// Column of element d of head h in a math warp's combine slot [GMAX][D]:
// the tensor-core write_comb stores one element per lane and instruction,
// and the bits of d flipped here put those 32 stores in 32 distinct banks.
// The combine reads 32 consecutive d of one head, which the flip permutes
// within their 32-element window (no conflict either).
template <bool MMA, int QK>
__device__ __forceinline__ int comb_col(int h, int d) {
    if constexpr (!MMA)
        return d;
    else if constexpr (QK != 0)   // lane (g, t) stores d = 16g + 2mt (+1), head 2t (+1) + 8nt
        return d ^ ((((d >> 5) & 3) << 2) | ((h >> 1) & 3));
    else                          // lane (g, t) stores d = 16mt + g (+8), head 2t (+1) + 8nt
        return d ^ (((h >> 1) & 3) << 3);
}

// ---------------------------------------------------------------------------
// consumer state
// ---------------------------------------------------------------------------
template <typename T, int D, int GMAX, bool MMA, int QK = 0>
struct Consumer;

// CUDA-core math: lane owns EPL = D/32 consecutive elements of head_dim.
template <typename T, int D, int GMAX>
struct Consumer<T, D, GMAX, false, 0> {
    static constexpr int EPL = D / 32;
    static constexpr int TB = GMAX <= 2 ? 16 : (GMAX == 4 ? 8 : (GMAX == 8 ? 4 : 2));
    static constexpr int LOGTB = TB == 16 ? 4 : (TB == 8 ? 3 : (TB == 4 ? 2 : 1));
    float qf[GMAX][EPL];
    float m[GMAX], l[GMAX];
    float acc[GMAX][EPL];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            m[h] = -CUDART_INF_F;
            l[h] = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
        }
    }

    __device__ __forceinline__ void load_q(const uint8_t *qslot, int gca, float scale_log2,
                                           int lane) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const T *row = reinterpret_cast<const T *>(qslot + h * D * sizeof(T));
                qf[h][e] = (h < gca) ? Elem<T>::to_f32(row[lane * EPL + e]) * scale_log2 : 0.f;
            }
        }
    }

    // lane's token within a batch after the reduce-scatter, and the inverse
    static __device__ __forceinline__ int token_of_lane(int lane) {
        int t = 0;
#pragma unroll
        for (int k = 0; k < LOGTB; ++k) t |= ((lane >> (4 - k)) & 1) << (LOGTB - 1 - k);
        return t;
    }
    static __device__ __forceinline__ int lane_of_token(int t) {
        int ln = 0;
#pragma unroll
        for (int k = 0; k < LOGTB; ++k) ln |= ((t >> (LOGTB - 1 - k)) & 1) << (4 - k);
        return ln;
    }

    __device__ __forceinline__ void tile(uint32_t sK, uint32_t sV, int ntok, int warp, int lane) {
        const int chunk = (lane * EPL * (int)sizeof(T)) >> 4;
        const int within = (lane * EPL * (int)sizeof(T)) & 15;
        const int tl = token_of_lane(lane);
#pragma unroll 1
        for (int b0 = 0; b0 < 16; b0 += TB) {
            const int rbase = 16 * warp + b0;
            if (rbase >= ntok) break;
            // partial dots of this lane's head_dim slice for TB tokens
            float part[GMAX][TB];
#pragma unroll
            for (int t = 0; t < TB; ++t) {
                float kf[EPL];
                lds_vec<T, EPL>(swz(sK, rbase + t, chunk) + within, kf);
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) a = fmaf(qf[h][e], kf[e], a);
                    part[h][t] = a;
                }
            }
            // reduce-scatter over the warp: afterwards part[h][0] is the full
            // dot product of token tl (held by 32/TB lanes)
#pragma unroll
            for (int k = 0; k < LOGTB; ++k) {
                const int mask = 16 >> k;
                const bool up = (lane & mask) != 0;
                const int half = TB >> (k + 1);
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const float send = up ? part[h][i] : part[h][i + half];
                        const float keep = up ? part[h][i + half] : part[h][i];
                        part[h][i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
                    }
                }
            }
#pragma unroll
            for (int k = LOGTB; k < 5; ++k) {
#pragma unroll
                for (int h = 0; h < GMAX; ++h)
                    part[h][0] += __shfl_xor_sync(0xffffffffu, part[h][0], 16 >> k);
            }
            const bool valid = rbase + tl < ntok;
            float p[GMAX];
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                const float sc = valid ? part[h][0] : -CUDART_INF_F;
                float mx = sc;
#pragma unroll
                for (int k = 0; k < 5; ++k) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16 >> k));
                const float mn = fmaxf(m[h], mx);
                const float alpha = exp2f(m[h] - mn);
                p[h] = exp2f(sc - mn);
                float ps = p[h];
#pragma unroll
                for (int k = 0; k < LOGTB; ++k) ps += __shfl_xor_sync(0xffffffffu, ps, 16 >> k);
                l[h] = l[h] * alpha + ps;
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[h][e] *= alpha;
                m[h] = mn;
            }
            // P V
#pragma unroll
            for (int t = 0; t < TB; ++t) {
                if (rbase + t < ntok) {
                    float vf[EPL];
                    lds_vec<T, EPL>(swz(sV, rbase + t, chunk) + within, vf);
                    const int src = lane_of_token(t);
#pragma unroll
                    for (int h = 0; h < GMAX; ++h) {
                        const float pt = __shfl_sync(0xffffffffu, p[h], src);
#pragma unroll
                        for (int e = 0; e < EPL; ++e) acc[h][e] = fmaf(pt, vf[e], acc[h][e]);
                    }
                }
            }
        }
    }

    __device__ __forceinline__ void write_comb(float *comb_o, float *comb_m, float *comb_l,
                                               int warp, int lane) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            float *o = comb_o + (warp * GMAX + h) * D + lane * EPL;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] = acc[h][e];
            if (lane == 0) {
                comb_m[warp * GMAX + h] = m[h];
                comb_l[warp * GMAX + h] = l[h];
            }
        }
    }
};

// Tensor-core math: per warp, S^T[16 tokens x 8 heads] = K Q^T and
// O^T[D x 8 heads] += V^T P^T with mma.sync m16n8k16 (fp32 accumulate).
//
// 8-bit caches (QK != 0): codes go from shared memory straight into the mma
// fragments as exact fp16 values (every int8 and E4M3 value is one), with no
// 16-bit copy of the tile. Two index permutations make each thread's codes
// whole 16-byte chunks:
//  - S^T = K Q^T sums over d, so d may be renumbered in K and q alike: lane
//    (g, t) = (lane / 4, lane % 4) takes bytes [32t, 32t + 32) of K rows g and
//    g + 8, and k-step ks, k index {2t, 2t+1, 2t+8, 2t+9} stands for element
//    32t + 4ks + {0, 1, 2, 3}; load_q puts q in the same order.
//  - in O^T = V^T P^T the rows of O^T are d: row 16mt + g of m-tile mt stands
//    for element 16g + 2mt and row 16mt + g + 8 for 16g + 2mt + 1, so lane
//    (g, t) takes bytes [16g, 16g + 16) of V rows 2t, 2t+1, 2t+8, 2t+9 (the
//    tokens of its fragment); write_comb puts d back in order.
// Each q head is scaled by a power of two 2^-e (e >= 0) that keeps it below
// 2^15, and e is folded back into that head's score factor; the scaling is
// exact. The row scales enter as
//     score_t = s_k[t] * <q, code_k[t]>,
//     o = sum_t p_t s_v[t] code_v[t] / sum_t p_t,
// with s_v[t] / max(s_v of the warp's 16 rows) multiplied into p_t before
// it is split into fp16 parts (so it stays <= 1), and the running factor
// sigma (that maximum) carried beside the accumulator, which holds o / sigma.
template <typename T, int D, int GMAX, int QK>
struct Consumer<T, D, GMAX, true, QK> {
    using MT = typename std::conditional<QK != 0, __half, T>::type;  // mma operand type
    static constexpr int TT = tile_tokens(QK, GMAX);                  // rows of a tile
    static constexpr int NTN = GMAX / 8;
    static constexpr int KS = D / 16;
    uint32_t qb[NTN][KS][2];
    float acc[KS][NTN][4];
    float m[NTN][2], l[NTN][2];
    uint32_t pbuf;  // this warp's P staging buffer (NTN x {hi, lo} x 256 B)
    float scale_log2;
    float sl2[NTN][2];  // 8-bit caches: score factor of this thread's score heads
    float sigma;        // 8-bit caches: the accumulator holds o / sigma
    // int8 caches: kInt8Bias x sum_d q of this thread's score heads, and
    // kInt8Bias x sum_t p' over the warp's tokens of the last tile (the fp16
    // parts its PV product used), which that product left in the
    // accumulators of those heads. It comes off at the next tile's rescale
    // (or the segment's end): left to pile up over a segment, the bias, far
    // above the signal sum p' code, made the accumulators' rounding grow with
    // the segment's length (9e-4 on outputs of ~0.006 over 34k tokens).
    float qsb[NTN][2], pbias[NTN][2];

    __device__ __forceinline__ void reset() {
        sigma = 0.f;
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                m[nt][hh] = -CUDART_INF_F;
                l[nt][hh] = 0.f;
                pbias[nt][hh] = 0.f;
            }
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[ks][nt][i] = 0.f;
        }
    }

    __device__ __forceinline__ void load_q(const uint8_t *qslot, int gca, float sl2_in, int lane) {
        scale_log2 = sl2_in;
        const int h_in = lane >> 2;        // n index (q head within the n-tile)
        const int k_in = (lane & 3) * 2;   // k index pair
        if constexpr (QK == 0) {
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt) {
                const int h = nt * 8 + h_in;
                const uint32_t *row = reinterpret_cast<const uint32_t *>(qslot + h * D * sizeof(T));
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qb[nt][ks][0] = (h < gca) ? row[(ks * 16 + k_in) >> 1] : 0u;
                    qb[nt][ks][1] = (h < gca) ? row[(ks * 16 + 8 + k_in) >> 1] : 0u;
                }
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt) {
                const int h = nt * 8 + h_in;
                // lane (g, t) holds elements 32t .. 32t + 31 of head h (word w:
                // elements 32t + 2w, + 1); the four lanes of head h hold all D
                static_assert(D == 128, "8-bit caches take head_dim 128");
                uint32_t qw[16];
                const uint4 *row4 =
                    reinterpret_cast<const uint4 *>(qslot + h * D * sizeof(T)) + 4 * (lane & 3);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = h < gca ? row4[c] : make_uint4(0u, 0u, 0u, 0u);
                    qw[4 * c] = v.x;
                    qw[4 * c + 1] = v.y;
                    qw[4 * c + 2] = v.z;
                    qw[4 * c + 3] = v.w;
                }
                float amax = 0.f;
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const float2 x = Elem<T>::unpack2(qw[w]);
                    amax = fmaxf(amax, fmaxf(fabsf(x.x), fabsf(x.y)));
                }
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                // amax < 2^(F+1); scaling by 2^-e, e = max(0, F - 14), keeps |q| < 2^15
                const int F = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
                const int e = F > 14 ? F - 14 : 0;
                const float mul = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        // k indices {2t, 2t+1} (half 0), {2t+8, 2t+9} (half 1) stand
                        // for elements 32t + 4ks + 2half, + 1: word 2ks + half
                        const float2 x = Elem<T>::unpack2(qw[2 * ks + half]);
                        __half2 q2 = __floats2half2_rn(x.x * mul, x.y * mul);
                        qb[nt][ks][half] = *reinterpret_cast<uint32_t *>(&q2);
                    }
                // int8: sum of head h's fp16 q elements (the four lanes of h)
                float qs = 0.f;
                if constexpr (QK == kQuantInt8) {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const float2 x = __half22float2(
                                *reinterpret_cast<const __half2 *>(&qb[nt][ks][half]));
                            qs += x.x + x.y;
                        }
                    qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                    qs += __shfl_xor_sync(0xffffffffu, qs, 2);
                }
                // score heads of this thread: 8nt + 2(lane%4) + hh, whose shift
                // (and q sum) sits with lanes 4 * (2(lane%4) + hh)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int src = ((lane & 3) * 2 + hh) * 4;
                    const int es = __shfl_sync(0xffffffffu, e, src);
                    sl2[nt][hh] = scale_log2 * __uint_as_float((uint32_t)(127 + es) << 23);
                    if constexpr (QK == kQuantInt8)
                        qsb[nt][hh] = kInt8Bias * __shfl_sync(0xffffffffu, qs, src);
                }
            }
        }
    }

    // 8-bit caches: sK / sV hold codes, ksc / vsc (shared addresses) the
    // tile's K and V row scales
    __device__ __forceinline__ void tile(uint32_t sK, uint32_t sV, int ntok, int warp, int lane,
                                         uint32_t ksc = 0, uint32_t vsc = 0) {
        const int r0 = 16 * warp;
        const int nval = ntok - r0;
        if (nval <= 0) return;
        const int g = lane >> 2, t = lane & 3;
        // 8-bit caches: all of this lane's codes of the tile, K then V, are
        // loaded before any is used (16-byte chunks; a quarter-warp's eight
        // chunks fall in distinct bank groups under the swizzle)
        uint32_t kw[2][8], vw[4][4];
        if constexpr (QK != 0) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    lds_u32x4(swz<TT>(sK, r0 + g + 8 * rr, 2 * t + c), kw[rr][4 * c], kw[rr][4 * c + 1],
                              kw[rr][4 * c + 2], kw[rr][4 * c + 3]);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                lds_u32x4(swz<TT>(sV, r0 + 2 * t + (k & 1) + 8 * (k >> 1), g), vw[k][0], vw[k][1],
                          vw[k][2], vw[k][3]);
        }
        const int rA = r0 + g, rB = rA + 8;   // this lane's score rows (tokens)
        const bool vA = rA < ntok, vB = rB < ntok;
        // 8-bit caches: row scales of K (into the scores) and V (into p); the
        // V side does not wait for the scores
        float ksA = 1.f, ksB = 1.f, fvA = 1.f, fvB = 1.f, ratio = 1.f;
        if constexpr (QK != 0) {
            ksA = vA ? lds_f32(ksc + 4 * rA) : 0.f;
            ksB = vB ? lds_f32(ksc + 4 * rB) : 0.f;
            const float vsA = vA ? lds_f32(vsc + 4 * rA) : 0.f;
            const float vsB = vB ? lds_f32(vsc + 4 * rB) : 0.f;
            float vmax = fmaxf(vsA, vsB);
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 4));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 8));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 16));
            if (!(vmax > 0.f)) vmax = 1.f;   // all-zero V rows: p' = 0 whatever vmax is
            const float inv = __frcp_rn(vmax);
            fvA = vsA * inv;
            fvB = vsB * inv;
            ratio = sigma * inv;             // the accumulator moves from o/sigma to o/vmax
            sigma = vmax;
        }
        // ---- S^T = K Q^T
        float s[NTN][4];
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
        if constexpr (QK != 0) {
            // even and odd k-steps in two accumulators: two chains of KS/2 mmas
            float s2[NTN][4];
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s2[nt][i] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a0, a1, a2, a3;
                codes_to_f16<QK>(kw[0][ks], a0, a2);   // row g:     k 2t, 2t+1 | 2t+8, 2t+9
                codes_to_f16<QK>(kw[1][ks], a1, a3);   // row g + 8
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt)
                    MmaOp<MT>::run((ks & 1) ? s2[nt] : s[nt], a0, a1, a2, a3, qb[nt][ks][0],
                                   qb[nt][ks][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s[nt][i] += s2[nt][i];
        } else {
            // even and odd k-steps in two accumulators: two chains of KS/2 mmas
            float s2[NTN][4];
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s2[nt][i] = 0.f;
            const int row = r0 + (lane & 15);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int chunk = ks * 2 + (lane >> 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(swz<TT>(sK, row, chunk), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt)
                    MmaOp<MT>::run((ks & 1) ? s2[nt] : s[nt], a0, a1, a2, a3, qb[nt][ks][0],
                                   qb[nt][ks][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) s[nt][i] += s2[nt][i];
        }

        // ---- online softmax (tokens rA, rB; heads 8nt + 2*(lane%4) + hh)
        float p[NTN][4];
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float fa = QK != 0 ? ksA * sl2[nt][hh] : scale_log2;
                const float fb = QK != 0 ? ksB * sl2[nt][hh] : scale_log2;
                float sva = s[nt][hh], svb = s[nt][2 + hh];
                if constexpr (QK == kQuantInt8) {   // the codes' bias off the scores
                    sva -= qsb[nt][hh];
                    svb -= qsb[nt][hh];
                }
                const float sa = vA ? sva * fa : -CUDART_INF_F;
                const float sb = vB ? svb * fb : -CUDART_INF_F;
                float mx = fmaxf(sa, sb);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const float mn = fmaxf(m[nt][hh], mx);
                const float alpha = exp2f(m[nt][hh] - mn);
                m[nt][hh] = mn;
                p[nt][hh] = exp2f(sa - mn);
                p[nt][2 + hh] = exp2f(sb - mn);
                l[nt][hh] = l[nt][hh] * alpha + p[nt][hh] + p[nt][2 + hh];
                const float ar = QK != 0 ? alpha * ratio : alpha;
                if constexpr (QK == kQuantInt8) {
                    // (acc - the last tile's bias) * ar, in one fma
                    const float nb = -pbias[nt][hh] * ar;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        acc[ks][nt][hh] = fmaf(acc[ks][nt][hh], ar, nb);
                        acc[ks][nt][2 + hh] = fmaf(acc[ks][nt][2 + hh], ar, nb);
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        acc[ks][nt][hh] *= ar;
                        acc[ks][nt][2 + hh] *= ar;
                    }
                }
                if constexpr (QK != 0) {   // p' = p * s_v / vmax for the PV product
                    p[nt][hh] *= fvA;
                    p[nt][2 + hh] *= fvB;
                }
            }
        }
        // ---- P^T as the B operand: stage [token][head] hi/lo pairs, reload transposed
        __syncwarp();
        uint32_t bh[NTN][2], bl[NTN][2];
        float psum[NTN][2];   // int8: this lane's share of sum_t p' per head
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
            const uint32_t hi = pbuf + nt * 512, lo = hi + 256;
            float r00, r01, r10, r11;
            const uint32_t hA = Elem<MT>::pack2(p[nt][0], p[nt][1], r00, r01);
            const uint32_t hB = Elem<MT>::pack2(p[nt][2], p[nt][3], r10, r11);
            float d00, d01, d10, d11;
            const uint32_t lA = Elem<MT>::pack2(p[nt][0] - r00, p[nt][1] - r01, d00, d01);
            const uint32_t lB = Elem<MT>::pack2(p[nt][2] - r10, p[nt][3] - r11, d10, d11);
            if constexpr (QK == kQuantInt8) {   // the p' values the product uses, per head
                psum[nt][0] = (r00 + d00) + (r10 + d10);
                psum[nt][1] = (r01 + d01) + (r11 + d11);
            }
            const uint32_t offA = (lane >> 2) * 16 + (lane & 3) * 4;
            const uint32_t offB = offA + 8 * 16;
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(hi + offA), "r"(hA) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(hi + offB), "r"(hB) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(lo + offA), "r"(lA) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(lo + offB), "r"(lB) : "memory");
        }
        __syncwarp();
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
            const uint32_t hi = pbuf + nt * 512, lo = hi + 256;
            ldsm_x2_t(hi + (lane & 15) * 16, bh[nt][0], bh[nt][1]);
            ldsm_x2_t(lo + (lane & 15) * 16, bl[nt][0], bl[nt][1]);
        }
        // ---- O^T += V^T P^T
        if constexpr (QK != 0) {
            // m-tile mt: rows g / g + 8 are elements 16g + 2mt / + 1, i.e.
            // byte 2mt / 2mt + 1 of the chunk; k = tokens 2t, 2t+1 (vw[0], vw[1])
            // and 2t+8, 2t+9 (vw[2], vw[3]), paired byte-wise
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    const int mt = 2 * i + hb;
                    const uint32_t sel = hb ? 0x7362u : 0x5140u;
                    uint32_t z01, z23, a0, a1, a2, a3;
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(z01) : "r"(vw[0][i]), "r"(vw[1][i]), "r"(sel));
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(z23) : "r"(vw[2][i]), "r"(vw[3][i]), "r"(sel));
                    codes_to_f16<QK>(z01, a0, a1);
                    codes_to_f16<QK>(z23, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NTN; ++nt) {
                        MmaOp<MT>::run(acc[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
                        MmaOp<MT>::run(acc[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
                    }
                }
            if constexpr (QK == kQuantInt8) {
                // this tile's bias: the eight lanes' shares of each head
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float b = psum[nt][hh];
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) b += __shfl_xor_sync(0xffffffffu, b, o);
                        pbias[nt][hh] = kInt8Bias * b;
                    }
            }
        } else {
            const int tok = r0 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int chunk = mt * 2 + ((lane >> 3) & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(swz<TT>(sV, tok, chunk), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt) {
                    MmaOp<MT>::run(acc[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
                    MmaOp<MT>::run(acc[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
                }
            }
        }
        __syncwarp();  // P buffer reads done before the next tile rewrites it
    }

    __device__ __forceinline__ void write_comb(float *comb_o, float *comb_m, float *comb_l,
                                               int warp, int lane) {
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float lt = l[nt][hh];
                lt += __shfl_xor_sync(0xffffffffu, lt, 4);
                lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                lt += __shfl_xor_sync(0xffffffffu, lt, 16);
                const int h = nt * 8 + (lane & 3) * 2 + hh;
                if (lane < 4) {
                    comb_m[warp * GMAX + h] = m[nt][hh];
                    comb_l[warp * GMAX + h] = lt;
                }
            }
            const float sg = QK != 0 ? sigma : 1.f;
            // int8: the last tile's bias of heads 2(lane%4) and + 1
            float b0 = 0.f, b1 = 0.f;
            if constexpr (QK == kQuantInt8) {
                b0 = pbias[nt][0];
                b1 = pbias[nt][1];
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int h = nt * 8 + (lane & 3) * 2;
                // rows g and g + 8 of m-tile mt hold elements d and d + dd
                const int d = QK != 0 ? 16 * (lane >> 2) + 2 * mt : mt * 16 + (lane >> 2);
                const int dd = QK != 0 ? 1 : 8;
                float *o = comb_o + (warp * GMAX + h) * D;
                o[comb_col<true, QK>(h, d)] = (acc[mt][nt][0] - b0) * sg;
                o[D + comb_col<true, QK>(h + 1, d)] = (acc[mt][nt][1] - b1) * sg;
                o[comb_col<true, QK>(h, d + dd)] = (acc[mt][nt][2] - b0) * sg;
                o[D + comb_col<true, QK>(h + 1, d + dd)] = (acc[mt][nt][3] - b1) * sg;
            }
        }
    }
};

// ---------------------------------------------------------------------------
// E4M3 codes on the 5th-generation tensor cores (tcgen05)
// ---------------------------------------------------------------------------
// x rounded to 4 significant bits (half away from zero): half of the 20
// dropped mantissa bits added, then those bits cleared. Every value of 4
// significant bits in E4M3's normal range is an E4M3 value.
__device__ __forceinline__ float round_sig4(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x80000u) & 0xFFF00000u);
}

// x = x1 + x2 / 16 + x3 / 256 + e, |e| <= 2^-12 |x| (E4M3 normal range), with
// x1, x2 of 4 significant bits; x3 is left for the E4M3 conversion to round.
__device__ __forceinline__ void e4m3_parts(float x, float &x1, float &x2, float &x3) {
    x1 = round_sig4(x);
    const float r1 = __fmul_rn(__fsub_rn(x, x1), 16.f);
    x2 = round_sig4(r1);
    x3 = __fmul_rn(__fsub_rn(r1, x2), 16.f);
}

// two fp32 to E4M3 codes (round to nearest, saturating): a in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Heads h0 .. h0 + 3 of x as their three E4M3 parts each, byte 3i + j for
// part j of head h0 + i; bytes 12..15 are 0.
template <int GMAX>
__device__ __forceinline__ uint4 pack_parts4(const float (&x)[GMAX], int h0) {
    float v[12];
#pragma unroll
    for (int i = 0; i < 4; ++i) e4m3_parts(x[h0 + i], v[3 * i], v[3 * i + 1], v[3 * i + 2]);
    uint32_t w[3];
#pragma unroll
    for (int q = 0; q < 3; ++q)
        w[q] = e4m3x2(v[4 * q], v[4 * q + 1]) | (e4m3x2(v[4 * q + 2], v[4 * q + 3]) << 16);
    return make_uint4(w[0], w[1], w[2], 0u);
}

// Largest of v_i over the warp for i = lane / 8, the four values reduced
// together: the first exchange halves the values each lane holds, the second
// halves them again, and three more finish the reduction (6 shuffles, not 20).
__device__ __forceinline__ float warp_max4(float v0, float v1, float v2, float v3, int lane) {
    const bool hi16 = lane & 16, hi8 = lane & 8;
    float a = hi16 ? v2 : v0, b = hi16 ? v3 : v1;   // kept
    const float c = hi16 ? v0 : v2, d = hi16 ? v1 : v3;
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, c, 16));
    b = fmaxf(b, __shfl_xor_sync(0xffffffffu, d, 16));
    float e = hi8 ? b : a;
    e = fmaxf(e, __shfl_xor_sync(0xffffffffu, hi8 ? a : b, 8));
    e = fmaxf(e, __shfl_xor_sync(0xffffffffu, e, 4));
    e = fmaxf(e, __shfl_xor_sync(0xffffffffu, e, 2));
    return fmaxf(e, __shfl_xor_sync(0xffffffffu, e, 1));
}

// The math warps form groups of four that take turns on the tiles of the
// CTA's range (tile i goes to group i % groups). In a group, thread r = 32 (warp % 4) + lane owns tensor-memory
// lane r: token r of the tile for the scores, element d = r of head_dim for
// the output. Per tile, one thread of the group issues
//   S = K Q^T   M = 128 tokens (the stage's K codes, K-major), N = 3 gca
//               columns (each q head as three E4M3 parts), K = 128 in 4 mmas,
//   O = V^T P   M = 128 elements (the stage's V codes, read M-major), N = 16
//               columns (four heads' p as three E4M3 parts each; a second
//               product for heads 4..7), K = 128 tokens in 4 mmas,
// both with fp32 accumulators in tensor memory. P is stored token-major
// without swizzle (16 bytes per token), so each thread writes its token's
// parts with one 16-byte store. q_h c_h = x1 + x2/16 + x3/256
// with E4M3 parts and c_h a power of two; p' = p s_v 256 / max s_v alike. The
// group keeps one running max per head (exchanged through shared memory each
// tile); each thread keeps its token's share of the sums l and its element's
// accumulators. The swizzled stage is the operands' layout as it is: rows of
// 128 bytes, 16-byte chunk c of row r at c ^ (r % 8), 1024-byte atoms.
template <typename T, int D, int GMAX>
struct TcConsumer {
    static_assert(D == 128 && (GMAX == 4 || GMAX == 8),
                  "tensor-core E4M3 path: head_dim 128, up to 4 or 8 heads");
    float m[GMAX], lp[GMAX], acc[GMAX], sl2[GMAX];
    int gca = 0, g = 0, qw = 0, r = 0;
    bool issuer = false;                 // the group's first warp
    bool wide = false, pv2 = false;      // scores on 32 columns (gca > 5); a second PV product (gca > 4)
    uint32_t idesc_qk = 0, idesc_pv = 0;
    uint64_t dq = 0;                     // descriptor of the q parts
    uint32_t nproc = 0, xph = 0;         // tiles processed; group barrier uses
    uint32_t tS = 0, tO = 0;             // this lane quarter's S and O columns
    uint32_t qp = 0, pb = 0, xbuf = 0, qsc = 0;
    uint32_t barS = 0, barO = 0, barX = 0, barP = 0;
    unsigned *err = nullptr;
    uint64_t wait_ns = 0;

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            m[h] = -CUDART_INF_F;
            lp[h] = 0.f;
            acc[h] = 0.f;
        }
    }

    // A bounded wait whose outcome is the whole warp's: the tcgen05 loads that
    // follow are .sync.aligned, so every lane goes on or every lane leaves.
    __device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
        const bool ok = mbar_wait(bar, parity, err, wait_ns);
        return __all_sync(0xffffffffu, ok);
    }

    // barrier of the group's four warps (mbarrier, bounded)
    __device__ __forceinline__ bool gsync(int lane) {
        __syncwarp();
        if (lane == 0) mbar_arrive(barX);
        const bool ok = warp_wait(barX, xph & 1u);
        ++xph;
        return ok;
    }

    // The unit's q heads as E4M3 parts: rows 3h + j of this group's B operand
    // (K-major, 128-byte swizzle), and each head's score factor.
    __device__ __forceinline__ bool first(const uint8_t *qslot, int gca_, float scale_log2,
                                          int lane) {
        reset();
        gca = gca_;
        wide = GMAX > 4 && 3 * gca > 16;
        pv2 = GMAX > 4 && gca > 4;
        idesc_qk = idesc_e4m3(128, wide ? 32 : 16, false, false);
        idesc_pv = idesc_e4m3(128, 16, true, true);
        dq = sdesc_sw128(qp, 16, 1024);
        // warp qw takes heads hb + qw (hb = 0, 4): lane t holds elements
        // 4t .. 4t + 3, so a head's largest element is one warp reduction
#pragma unroll
        for (int hb = 0; hb < GMAX; hb += 4) {
            const int h = hb + qw;   // warp-uniform
            if (h >= gca) break;
            const uint2 v =
                *reinterpret_cast<const uint2 *>(qslot + (size_t)h * D * sizeof(T) + lane * 8);
            const float2 f0 = Elem<T>::unpack2(v.x), f1 = Elem<T>::unpack2(v.y);
            const float x[4] = {f0.x, f0.y, f1.x, f1.y};
            const float amax =
                warp_max_f32(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
            // amax in [2^F, 2^(F+1)): c = 2^E, E = 7 - F, puts the head's largest
            // element in [128, 256); E is clamped so that c and 1/c stay normal
            const int F = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
            const int E = max(-120, min(120, 7 - F));
            const float c = __uint_as_float((uint32_t)(127 + E) << 23);
            float p1[4], p2[4], p3[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) e4m3_parts(x[k] * c, p1[k], p2[k], p3[k]);
            const uint32_t b[3] = {e4m3x2(p1[0], p1[1]) | (e4m3x2(p1[2], p1[3]) << 16),
                                   e4m3x2(p2[0], p2[1]) | (e4m3x2(p2[2], p2[3]) << 16),
                                   e4m3x2(p3[0], p3[1]) | (e4m3x2(p3[2], p3[3]) << 16)};
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int n = 3 * h + j;
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(qp + n * 128 +
                                                              ((((lane >> 2) ^ (n & 7))) << 4) +
                                                              (lane & 3) * 4),
                             "r"(b[j])
                             : "memory");
            }
            if (lane == 0) sts_f32(qsc + 4 * h, __uint_as_float((uint32_t)(127 - E) << 23));
        }
        fence_proxy_async_smem();
        if (!gsync(lane)) return false;
#pragma unroll
        for (int hh = 0; hh < GMAX; ++hh) sl2[hh] = hh < gca ? scale_log2 * lds_f32(qsc + 4 * hh) : 0.f;
        return true;
    }

    // column c of the loaded S or O values
    __device__ __forceinline__ static float col(const uint32_t (&a)[16], const uint32_t (&b)[16],
                                                int c) {
        return __uint_as_float(c < 16 ? a[c] : b[c - 16]);
    }

    __device__ __forceinline__ bool tile(uint32_t sK, uint32_t sV, uint32_t ksc, uint32_t vsc,
                                         int ntok, int lane) {
        const uint32_t ph = nproc & 1u;
        // ---- S = K Q^T: the issuing warp builds the (warp-uniform)
        // descriptors, one elected lane issues. (Issuing the group's next
        // tile's product right after this tile's PV product, when its stage
        // was full, made the llama-shaped step slower: 69.2 -> 77.8 us.)
        if (issuer) {
            // K step k: 32 bytes further along each 128-byte row (start field + 2k)
            const uint64_t dk = sdesc_sw128(sK, 16, 1024);
            if (elect_one()) {
                fence_proxy_async_smem();   // the stage's data, seen complete through its barrier
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k) tc_mma_e4m3(tS, dk + 2 * k, dq + 2 * k, idesc_qk, k);
                tc_commit(barS);
            }
        }
        __syncwarp();
        if (!warp_wait(barS, ph)) return false;
        tc_fence_after();
        uint32_t a[16], b[16];
        tmem_ld16(tS, a);
        if (wide) tmem_ld16(tS + 16, b);
        tmem_ld_wait(a);
        if (wide) tmem_ld_wait(b);
        const bool valid = r < ntok;
        const float ks = lds_f32(ksc + 4 * r);
        const float vs = lds_f32(vsc + 4 * r);
        float s[GMAX];
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            const float v = col(a, b, 3 * h) + col(a, b, 3 * h + 1) * 0.0625f +
                            col(a, b, 3 * h + 2) * 0.00390625f;
            s[h] = (valid && h < gca) ? v * ks * sl2[h] : -CUDART_INF_F;
        }
        // ---- the group's max of each head's scores and of the V row scales:
        // this warp's maxima to the exchange slot (heads 4j .. 4j + 3 reduced
        // together; lane 8i then holds head 4j + i)
        constexpr int XS = GMAX <= 4 ? 32 : 64;   // exchange slot of one warp
        const uint32_t slot = xbuf + (xph & 1u) * 4 * XS + qw * XS;
        const float m03 = warp_max4(s[0], s[1], s[2], s[3], lane);
        const float vmx = warp_max_f32(valid ? vs : 0.f);
        if ((lane & 7) == 0) sts_f32(slot + 4 * (lane >> 3), m03);
        if constexpr (GMAX > 4) {
            if (pv2) {
                const float m47 = warp_max4(s[4], s[5], s[6], s[7], lane);
                if ((lane & 7) == 0) sts_f32(slot + 16 + 4 * (lane >> 3), m47);
            }
        }
        if (lane == 0) sts_f32(slot + 4 * GMAX, vmx);
        if (!gsync(lane)) return false;
        const uint32_t slot0 = slot - qw * XS;
        float M[GMAX + 1];
#pragma unroll
        for (int h = 0; h <= GMAX; ++h) {
            M[h] = -CUDART_INF_F;
            if (h < GMAX && h >= gca) continue;
#pragma unroll
            for (int w = 0; w < 4; ++w) M[h] = fmaxf(M[h], lds_f32(slot0 + w * XS + 4 * h));
        }
        float VM = M[GMAX];
        if (!(VM > 0.f)) VM = 1.f;   // all-zero V rows: p' = 0 whatever VM is
        const float vf = vs * __frcp_rn(VM) * 256.f;
        // ---- online softmax; token r's p' parts: 16 bytes (heads 0..3) at
        // pb + 16 r, and heads 4..7 at pb + 2048 + 16 r
        float alpha[GMAX], x[GMAX];
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            alpha[h] = 1.f;
            x[h] = 0.f;
            if (h >= gca) continue;
            const float mn = fmaxf(m[h], M[h]);
            alpha[h] = ex2_approx(m[h] - mn);
            m[h] = mn;
            const float p = valid ? ex2_approx(s[h] - mn) : 0.f;
            lp[h] = lp[h] * alpha[h] + p;
            x[h] = p * vf;
        }
        sts_u32x4(pb + 16 * r, pack_parts4(x, 0));
        if constexpr (GMAX > 4)
            if (pv2) sts_u32x4(pb + 2048 + 16 * r, pack_parts4(x, 4));
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(barP);
        // ---- O = V^T P'
        if (issuer) {
            if (!warp_wait(barP, ph)) return false;
            // K step k: tokens 32k..: V 4 atoms (4096 bytes) further, P 512 bytes
            const uint64_t dv = sdesc_sw128(sV, 1024, 1024), dp = sdesc_none(pb, 128);
            if (elect_one()) {
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k) tc_mma_e4m3(tO, dv + 256 * k, dp + 32 * k, idesc_pv, k);
                if (pv2)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma_e4m3(tO + 16, dv + 256 * k, dp + 128 + 32 * k, idesc_pv, k);
                tc_commit(barO);
            }
            __syncwarp();
        }
        if (!warp_wait(barO, ph)) return false;
        tc_fence_after();
        tmem_ld16(tO, a);
        if (pv2) tmem_ld16(tO + 16, b);
        tmem_ld_wait(a);
        if (pv2) tmem_ld_wait(b);
        const float of = VM * (1.f / 256.f);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            if (h >= gca) continue;
            const int c0 = h < 4 ? 3 * h : 16 + 3 * (h - 4);   // O columns of head h
            const float o = col(a, b, c0) + col(a, b, c0 + 1) * 0.0625f +
                            col(a, b, c0 + 2) * 0.00390625f;
            acc[h] = fmaf(acc[h], alpha[h], o * of);
        }
        tc_fence_before();
        ++nproc;
        return true;
    }

    // the group's state for the segment: m (the same in all four warps), this
    // warp's share of l, and the group's output (entry g)
    __device__ __forceinline__ void write_comb(float *comb_o, float *comb_m, float *comb_l,
                                               int warp, int lane) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            float l = lp[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            if (lane == 0) {
                comb_m[warp * GMAX + h] = m[h];
                comb_l[warp * GMAX + h] = l;
            }
            comb_o[(g * GMAX + h) * D + r] = acc[h];
        }
    }
};

// ---------------------------------------------------------------------------
// log-sum-exp merge of one warp's slice of a unit cut by CTA boundaries
// ---------------------------------------------------------------------------
// The partials of the unit come from CTAs c_first .. c_last (those with an
// empty tile range hold none); the first of them used slot
// pkv_partial_slot(c_first, ...), the later ones slot 0. With the partials'
// log2-sum-exp2 values lse_p and normalised outputs o_p,
//     lse = log2 sum_p 2^{lse_p},   out = sum_p 2^{lse_p - lse} o_p,
// taken in CTA order with a running maximum (one pass). Loads bypass L1: the
// other CTAs' slices were written during this launch.
// Where a unit's results go. Plain launches: the out rows of sequence s.
// Prefix-aware launches: head j of a prefix unit belongs to member
// members[m0 + j / G] (head h0 + j % G) and goes to that member's prefix
// result row, or straight to out when the member's context ends with the
// prefix; a grouped sequence's own unit goes to its suffix result rows.
struct UnitDest {
    int kind;   // 0 out rows of sequence s, 1 prefix unit (members), 2 suffix rows of s
    int s;      // kinds 0, 2
    int m0;     // kind 1
};

// Store element (head j, d) of a unit's result and its head's log2-sum-exp2:
// for out, with the element d == 0; for a result row, one copy per merge
// slice (elements idx = j D + d with idx % 128 in [32 w, 32 w + 32) form slice
// w), written with the slice's first element of the head, so that the slice's
// merge needs nothing another warp wrote.
template <int D>
__device__ __forceinline__ void put_result(const DecodeParams &p, const UnitDest &u, int h0, int j,
                                           int d, float o, float lse, const int16_t *members,
                                           const int *seq_len, int nv) {
    int s = u.s, h = h0 + j, dest = u.kind;
    if (u.kind == 1) {
        s = members[u.m0 + j / p.G];
        h = h0 + j % p.G;
        dest = seq_len[nv + s] == 0 ? 0 : 1;
    }
    const size_t row = (size_t)s * p.Hq + h;
    if (dest == 0) {
        store_out(p.out, row * D + d, p.out_dtype, o);
        if (p.lse_out && d == 0) p.lse_out[row] = lse;
    } else {
        const size_t r = (size_t)(dest - 1) * p.S * p.Hq + row;
        p.pb.res_o[r * D + d] = o;
        if ((d & 31) == 0) p.pb.res_l[r * kMergeSlices + (((j * D + d) & 127) >> 5)] = lse;
    }
}

// Count this warp's pending result slices: slice `warp` of each (sequence,
// kv head) entry of its list (elements idx = 32 warp + lane + 128 k of the
// kv group's G x D outputs). A slice whose count reaches 2 (the prefix
// result's and the suffix result's slice are in) is merged by this warp into
// out: out = (2^{l_P} o_P + 2^{l_S} o_S) / (2^{l_P} + 2^{l_S}), up to 16
// elements per lane with their loads in flight together.
template <int D>
__device__ __forceinline__ void flush_final(const DecodeParams &p, int *list, int &n, int warp,
                                            int lane) {
    __syncwarp();
    const int e = lane < n ? list[lane] : 0;
    fence_acq_rel_gpu();
    unsigned prev = 0u;
    unsigned *cnt = p.pb.fin + (size_t)e * kMergeSlices + warp;
    if (lane < n) prev = atomicAdd(cnt, 1u);
    fence_acq_rel_gpu();
    const bool mine = lane < n && prev == 1u;
    const unsigned done = __ballot_sync(0xffffffffu, mine);
    __syncwarp();
    if (mine) {
        *cnt = 0u;   // both arrivals are in: reset for the next call
        // the finished entries' first output rows, compacted into the list
        const int sq = e / p.Hk, g = e - (e / p.Hk) * p.Hk;
        list[__popc(done & ((1u << lane) - 1u))] = sq * p.Hq + g * p.G;
    }
    __syncwarp();
    const int GD = p.G * D;
    const int ksv = (GD - 32 * warp + 127) / 128;   // this slice's elements per lane (at most)
    const int total = __popc(done) * ksv;
    const size_t plane = (size_t)p.S * p.Hq;
    for (int i0 = 0; i0 < total; i0 += 16) {
        float lp[16], ls[16], op[16], os[16];
        size_t row[16];
        int dd[16];
        bool ok[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const int it = i0 + t;
            const int b = it < total ? it / ksv : 0, k = it - b * ksv;
            const int idx = 32 * warp + lane + 128 * k;
            ok[t] = it < total && idx < GD;
            const int j = idx / D;
            dd[t] = idx - j * D;
            row[t] = (size_t)list[b] + j;
            if (ok[t]) {
                lp[t] = __ldcg(p.pb.res_l + row[t] * kMergeSlices + warp);
                ls[t] = __ldcg(p.pb.res_l + (plane + row[t]) * kMergeSlices + warp);
                op[t] = __ldcg(p.pb.res_o + row[t] * D + dd[t]);
                os[t] = __ldcg(p.pb.res_o + (plane + row[t]) * D + dd[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            if (!ok[t]) continue;
            const float m = fmaxf(lp[t], ls[t]);
            const float wp = exp2f(lp[t] - m), ws = exp2f(ls[t] - m);
            store_out(p.out, row[t] * D + dd[t], p.out_dtype, (wp * op[t] + ws * os[t]) / (wp + ws));
            if (p.lse_out && dd[t] == 0) p.lse_out[row[t]] = m + log2f(wp + ws);
        }
    }
    __syncwarp();
    n = 0;
}

// Note the (sequence, kv head) entries whose prefix or suffix result this
// warp has just written a slice of.
template <int D>
__device__ __forceinline__ void note_final(const DecodeParams &p, const UnitDest &u, int h0,
                                           int gca, const int16_t *members, const int *seq_len,
                                           int nv, int *list, int &n, int warp, int lane) {
    const int g = h0 / p.G;
    const int cnt = u.kind == 1 ? gca / p.G : 1;
    for (int m = 0; m < cnt; ++m) {
        const int s = u.kind == 1 ? members[u.m0 + m] : u.s;
        if (u.kind == 1 && seq_len[nv + s] == 0) continue;   // written to out directly
        if (lane == 0) list[n] = s * p.Hk + g;
        if (++n == kFinCap) flush_final<D>(p, list, n, warp, lane);
    }
}

// A cut segment waiting to be counted, with the facts of its unit's split
// (computed when the segment ends, so that the CTA's last moments do no
// 64-bit divisions): the CTAs c_first .. c_last holding its partials, their
// number, and the partial slot of CTA c_first.
// The work list may have two sections (prefix-aware launches: the prefix
// units, then every sequence's own units), each split over the C CTAs on its
// own, so that every CTA gets an equal share of both kinds of tile. Section k
// covers tiles [base, base + nt); a CTA's partial slots 2k and 2k + 1 serve
// it, and its arrival counters follow those of section 0 (c + k C).
struct PendSeg {
    TileMeta mt;
    int c_first, c_last, parts, slot_first;
};
// prefix-aware launches also keep the unit's section and where its results go
struct PendSegPfx : PendSeg {
    int sec;        // section of the unit
    int64_t nt;     // tiles of that section
    UnitDest ud;
};
template <bool PFX>
using PendSegT = typename std::conditional<PFX, PendSegPfx, PendSeg>::type;

// section of global tile tau: NT0 tiles in section 0 when there are two
// sections (NT0 > 0), else one section of NT tiles
__device__ __forceinline__ int section_of(int64_t tau, int64_t NT0, int64_t NT, int64_t &base,
                                          int64_t &nt) {
    const int k = (NT0 > 0 && tau >= NT0) ? 1 : 0;
    base = k ? NT0 : 0;
    nt = NT0 > 0 ? (k ? NT - NT0 : NT0) : NT;
    return k;
}

__device__ __forceinline__ PendSeg pend_seg(const TileMeta &mt, int C, int64_t NT) {
    PendSeg ps;
    ps.mt = mt;
    ps.c_first = pkv_owner(mt.tu, C, NT);
    ps.c_last = pkv_owner((int64_t)mt.tu + mt.nu - 1, C, NT);
    ps.parts = pkv_unit_parts(mt.tu, mt.nu, C, NT);
    ps.slot_first = pkv_partial_slot(ps.c_first, C, NT, mt.tu);
    return ps;
}

__device__ __forceinline__ PendSegPfx pend_seg_pfx(const TileMeta &mt, int C, int64_t NT0,
                                                   int64_t NT, const UnitDest &ud) {
    PendSegPfx ps;
    ps.mt = mt;
    ps.ud = ud;
    int64_t base, nt;
    ps.sec = section_of(mt.tu, NT0, NT, base, nt);
    ps.nt = nt;
    const int64_t tu = mt.tu - base;
    ps.c_first = pkv_owner(tu, C, nt);
    ps.c_last = pkv_owner(tu + mt.nu - 1, C, nt);
    ps.parts = pkv_unit_parts(tu, mt.nu, C, nt);
    ps.slot_first = pkv_partial_slot(ps.c_first, C, nt, tu) + 2 * ps.sec;
    return ps;
}

template <int D, int GMAX, int SLOTS, bool PFX>
__device__ __forceinline__ void merge_slice(const DecodeParams &p, const PendSegT<PFX> &ps,
                                            int warp, int lane, int64_t NT_all,
                                            const int16_t *members, const int *seq_len, int nv) {
    int64_t NT = NT_all;
    int sec = 0;
    if constexpr (PFX) {
        NT = ps.nt;
        sec = ps.sec;
    }
    const TileMeta &mt = ps.mt;
    const int c_first = ps.c_first;
    // the lane's elements are idx = warp*32 + lane + 128k, k < EPL, taken in
    // chunks of KC: all loads of one partial for a chunk are issued before
    // any of them is used, and at most KC elements are live at a time
    constexpr int EPL = (GMAX * D + kMergeSlices * 32 - 1) / (kMergeSlices * 32);
    constexpr int KC = EPL < 8 ? EPL : 8;
    const int C = p.C;
    const int n_el = mt.gca * D;
    const int c_last = ps.c_last;
    const int slot_first = ps.slot_first;
    const bool some_empty = NT < C;   // with NT >= C every CTA holds a tile
#pragma unroll 1
    for (int k0 = 0; k0 < EPL; k0 += KC) {
        if (warp * 32 + k0 * kMergeSlices * 32 >= n_el) break;
        float Mx[KC], W[KC], O[KC];
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            Mx[k] = -CUDART_INF_F;
            W[k] = 0.f;
            O[k] = 0.f;
        }
#pragma unroll 2
        for (int c = c_first; c <= c_last; ++c) {
            if (some_empty && pkv_cta_empty(c, C, NT)) continue;
            const int slot = c * SLOTS + (c == c_first ? slot_first : 2 * sec);
            // lane h < gca fetches this warp's copy of head h's lse
            const float lse_h =
                lane < mt.gca ? __ldcg(p.ws_lse + (slot * kMergeSlices + warp) * p.GC + lane)
                              : 0.f;
            float o[KC];
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                const int idx = warp * 32 + lane + (k0 + k) * kMergeSlices * 32;
                const int j = idx / D, d = idx - (idx / D) * D;
                o[k] = idx < n_el ? __ldcg(p.ws_o + (size_t)(slot * p.GC + j) * D + d) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                // head of element k0 + k: the same for every lane of the warp
                const int j = (warp * 32 + (k0 + k) * kMergeSlices * 32) / D;
                const float lse = __shfl_sync(0xffffffffu, lse_h, j & 31);
                const float mn = fmaxf(Mx[k], lse);
                const float a = exp2f(Mx[k] - mn), w = exp2f(lse - mn);
                W[k] = W[k] * a + w;
                O[k] = O[k] * a + w * o[k];
                Mx[k] = mn;
            }
        }
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            const int idx = warp * 32 + lane + (k0 + k) * kMergeSlices * 32;
            if (idx < n_el) {
                const int j = idx / D, d = idx - (idx / D) * D;
                if constexpr (PFX) {
                    put_result<D>(p, ps.ud, mt.h0, j, d, O[k] / W[k], Mx[k] + log2f(W[k]),
                                  members, seq_len, nv);
                } else {
                    store_out(p.out, ((size_t)mt.s * p.Hq + mt.h0 + j) * D + d, p.out_dtype,
                              O[k] / W[k]);
                    if (p.lse_out && d == 0)
                        p.lse_out[(size_t)mt.s * p.Hq + mt.h0 + j] = Mx[k] + log2f(W[k]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// fused append: the newest row into the stage's side slot
// ---------------------------------------------------------------------------
// Chunks i = tb, tb + tpb, ... < 2 * ROWB / 16 of row `row` ([S][Hk] rows of
// ROWB bytes) of k_new (i < ROWB / 16), then of v_new, to side + 16 i; zeros
// when !valid.
template <int ROWB>
__device__ __noinline__ void copy_new_row(uint32_t side, const void *k_new, const void *v_new,
                                          size_t row, int tb, int tpb, bool valid) {
    constexpr int CPR = ROWB / 16;
    const uint8_t *kn = static_cast<const uint8_t *>(k_new) + row * ROWB;
    const uint8_t *vn = static_cast<const uint8_t *>(v_new) + row * ROWB;
    for (int i = tb; i < 2 * CPR; i += tpb)
        cp_async_16(side + i * 16, i < CPR ? kn + i * 16 : vn + (i - CPR) * 16, valid);
}

// ---------------------------------------------------------------------------
// prefix-aware: the producers' jump to their range of the second section
// ---------------------------------------------------------------------------
// Out of line: the issue loop is unrolled and its code size shows in the
// instruction fetch.
static __device__ __noinline__ void cursor_jump(PkvCursor &c, int64_t tau, const int *seq_prefix,
                                                const int *seq_len, int W, int tt) {
    pkv_cursor_at(c, tau, seq_prefix, seq_len, W, tt);
}

// ---------------------------------------------------------------------------
// prefix-aware: the q rows of a prefix unit
// ---------------------------------------------------------------------------
// Row j of the unit is head h0 + j % G of member j / G (a sequence id from
// `members`); rows are QROWB bytes, copied in 16-byte chunks by the producer
// threads.
template <int QROWB>
__device__ __noinline__ void copy_q_members(uint32_t sQ, const void *q, const int16_t *members,
                                            int G, int Hq, int h0, int rows, int pt) {
    constexpr int CPRQ = QROWB / 16;
    const uint8_t *qb = static_cast<const uint8_t *>(q);
    for (int i = pt; i < rows * CPRQ; i += kProducerThreads) {
        const int j = i / CPRQ, c = i - (i / CPRQ) * CPRQ;
        const size_t row = (size_t)members[j / G] * Hq + h0 + j % G;
        cp_async_16(sQ + i * 16, qb + row * QROWB + c * 16, true);
    }
}

// ---------------------------------------------------------------------------
// fused append: write each context's newest K/V row into its slot
// ---------------------------------------------------------------------------
// Run by the producer threads of a CTA once they have issued their last
// tile. For every unit of chunk 0 whose last tile lies in this CTA's range
// [t_begin, t_end) (so exactly one CTA handles each (sequence, kv head)), the
// rows k_new[s][g] and v_new[s][g] go to position L - 1 of sequence s: block
// block_tables[s][(L - 1) / B], offset (L - 1) % B. The stores wait for the
// preceding kernel on the stream, like every store of the decode. A block id
// outside the pool is skipped (the tile loop has flagged it already).
template <typename Cfg>
__device__ __forceinline__ void fused_append_rows(const DecodeParams &p, const int *seq_prefix,
                                                  const int *seq_len, int64_t t_begin,
                                                  int64_t t_end, int pt, bool waited) {
    constexpr int CPR = Cfg::ROWB / 16;        // 16-byte chunks per row
    constexpr int CPU = 2 * CPR;               // K and V chunks per unit
    static_assert(kProducerThreads % CPU == 0, "a unit's chunks fill whole thread groups");
    constexpr int UPP = kProducerThreads / CPU;   // units per pass of the producer threads
    const int j = pt / CPU, c = pt - (pt / CPU) * CPU;
    const bool is_v = c >= CPR;
    const int ch = is_v ? c - CPR : c;
    PkvCursor cur;
    pkv_cursor_at(cur, t_begin, seq_prefix, seq_len, p.S, Cfg::TT);
    int k = 0;   // index of the unit end among this CTA's chunk-0 unit ends
    while (cur.s < p.S) {
        const int64_t T_u = (int64_t)seq_prefix[cur.s] + (int64_t)cur.u * cur.n;
        if (T_u >= t_end) break;
        const int64_t last = T_u + cur.n - 1;
        if (last >= t_end) break;   // the unit ends in a later CTA's range
        if (last >= t_begin && cur.u % p.NC == 0) {
            if (k % UPP == j) {
                if (!waited) {
                    grid_dependency_wait();
                    waited = true;
                }
                const int g = cur.u / p.NC;
                const int pos = cur.L - 1;
                const int e = __ldg(p.block_tables + (size_t)cur.s * p.M + pos / p.B);
                if (e >= 0 && e < p.NB) {
                    const size_t src = ((size_t)cur.s * p.Hk + g) * Cfg::ROWB + ch * 16;
                    const size_t dst = (((size_t)e * p.Hk + g) * p.B + pos % p.B) * Cfg::ROWB +
                                       ch * 16;
                    const uint8_t *from = static_cast<const uint8_t *>(is_v ? p.v_new : p.k_new);
                    uint8_t *to = static_cast<uint8_t *>(const_cast<void *>(is_v ? p.vp : p.kp));
                    *reinterpret_cast<uint4 *>(to + dst) =
                        __ldg(reinterpret_cast<const uint4 *>(from + src));
                }
            }
            ++k;
        }
        // next unit (skipping sequences without tiles)
        cur.ti = cur.n - 1;
        pkv_cursor_next(cur, seq_len, p.S, p.U, Cfg::TT);
    }
}

// ---------------------------------------------------------------------------
// the split-K kernel
// ---------------------------------------------------------------------------
template <typename T, int D, int GMAX, bool MMA, int QK, bool FLAT, bool FUSED, bool PFX>
__global__ void __launch_bounds__(kernel_threads(QK, GMAX), two_ctas(QK, GMAX, MMA, PFX) ? 2 : 1)
    decode_split_kernel(const DecodeParams p,
                        const typename std::conditional<PFX, PrefixMap, NoPrefixMap>::type pm) {
    using Cfg = SplitCfg<T, D, GMAX, MMA, QK, FUSED, PFX>;
    static_assert(!PFX || (MMA && QK == 0 && !FLAT && !FUSED), "prefix-aware: 16-bit paged mma");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    // TC scratch: exchange slots, q scales, the TMEM address, barriers
    const uint32_t tcx = (sbase + Cfg::OFF_TCX + 15u) & ~15u;
    const uint32_t tcbar = tcx + Cfg::TCX_BAR;
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + Cfg::OFF_META);
    const uint32_t full0 = sbase + Cfg::OFF_FULL;
    const uint32_t empty0 = sbase + Cfg::OFF_EMPTY;
    const uint32_t comb_full = sbase + Cfg::OFF_CBAR;
    const uint32_t comb_empty = comb_full + 8;
    float *comb_o = reinterpret_cast<float *>(smem + Cfg::OFF_COMB_O);
    float *comb_m = reinterpret_cast<float *>(smem + Cfg::OFF_COMB_M);
    float *comb_l = reinterpret_cast<float *>(smem + Cfg::OFF_COMB_L);
    // work sequences: the batch, preceded (prefix-aware) by the virtual prefix ones
    int nv = 0;
    if constexpr (PFX) nv = pm.nv;
    const int W = nv + p.S;
    int *seq_prefix = reinterpret_cast<int *>(smem + Cfg::OFF_SEQ);
    int *seq_len = seq_prefix + W + 1;
    int *seq_tab = seq_len + W;                       // prefix-aware only
    int16_t *members = reinterpret_cast<int16_t *>(seq_tab + W);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x, C = p.C;

    if (tid == 0) {
        for (int i = 0; i < Cfg::NST; ++i) {
            mbar_init(full0 + 8 * i, kProducerThreads + 1);
            mbar_init(empty0 + 8 * i, Cfg::CW);
        }
        mbar_init(comb_full, Cfg::CW);
        mbar_init(comb_empty, Cfg::TC ? 4 : Cfg::CW);   // TC: the merging group's warps
        if constexpr (Cfg::TC) {
            // per group: S done, O done (tcgen05.commit), the group's barrier,
            // p parts written; then TMEM allocated, TMEM no longer used
            const uint32_t tb = tcbar;
            for (int gi = 0; gi < Cfg::NG; ++gi) {
                mbar_init(tb + 8 * (0 * Cfg::NG + gi), 1);
                mbar_init(tb + 8 * (1 * Cfg::NG + gi), 1);
                mbar_init(tb + 8 * (2 * Cfg::NG + gi), 4);
                mbar_init(tb + 8 * (3 * Cfg::NG + gi), 4);
            }
            mbar_init(tb + 8 * (4 * Cfg::NG), 1);
            mbar_init(tb + 8 * (4 * Cfg::NG + 1), Cfg::CW);
        }
        fence_mbarrier_init();
    }
    // Inputs may come from the previous kernel on the stream (launched with
    // programmatic serialisation): wait for it before reading any of them.
    // With tables_ready the lengths and tables are complete already: they
    // are read (and the first table entries fetched) while that kernel runs,
    // and the wait comes just before q, the pools or any output is touched.
    if (!p.tables_ready) grid_dependency_wait();
    if constexpr (PFX)
        build_seq_arrays<FLAT, Cfg::TT, true>(p, W, seq_prefix, seq_len, cta == 0, pm, seq_tab,
                                              members);
    else
        build_seq_arrays<FLAT, Cfg::TT>(p, W, seq_prefix, seq_len, cta == 0);

    // zero-length sequences: zeros, written by CTA s % C (prefix-aware: not
    // the members of a group, whose output comes at least from the prefix)
    bool waited = !p.tables_ready;
    for (int s = 0; s < p.S; ++s) {
        bool empty = seq_len[nv + s] == 0;
        if constexpr (PFX) empty = empty && pm.w[nv + s].blocks == 0;
        if (empty && s % C == cta) {
            if (!waited) {   // the same for the whole CTA
                grid_dependency_wait();
                waited = true;
            }
            for (int i = tid; i < p.Hq * D; i += Cfg::THREADS)
                store_out(p.out, (size_t)s * p.Hq * D + i, p.out_dtype, 0.f);
            if (p.lse_out)
                for (int h = tid; h < p.Hq; h += Cfg::THREADS)
                    p.lse_out[(size_t)s * p.Hq + h] = -CUDART_INF_F;
        }
    }

    // this CTA's tiles: [b0, e0) of section 0 (prefix-aware: the prefix
    // units, NT0 tiles) and [b1, e1) of the rest; one section otherwise
    const int64_t NT = seq_prefix[W];
    const int64_t NT0 = PFX ? seq_prefix[nv] : 0, NT1 = NT - NT0;
    const int64_t b0 = NT0 ? pkv_split(cta, C, NT0) : 0, e0 = NT0 ? pkv_split(cta + 1, C, NT0) : 0;
    const int64_t b1 = NT0 + (NT1 ? pkv_split(cta, C, NT1) : 0);
    const int64_t e1 = NT0 + (NT1 ? pkv_split(cta + 1, C, NT1) : 0);
    const int n0 = (int)(e0 - b0);
    const int n_my = n0 + (int)(e1 - b1);
    const int64_t t_begin = n0 ? b0 : b1;
    constexpr int SLOTS = PFX ? 4 : 2;   // partial slots per CTA: two per section
    grid_dependents_launch();   // the next kernel on the stream may start its launch now
    if (n_my <= 0) return;

    if (warp >= Cfg::CW) {
        // ======================= producer warps =======================
        // 128 threads gather each tile with 16-byte cp.async copies straight
        // into the swizzled stage layout. Thread pt copies one physical block
        // of the tile (tpb threads per block), so it needs one block-table
        // entry per tile; entries are loaded LA tiles ahead into a register
        // ring whose slots are fixed by unrolling the loop LA times. Rows past
        // the context, blocks past the tile and out-of-pool block ids are
        // zero-filled (src-size 0): no address outside the pool is formed
        // and the math warps never see stale or garbage rows.
        // LA = 4: the loop body is unrolled LA times and its code size shows
        // in the instruction fetch (measured on the Llama-shaped step: 8 tiles
        // ahead 118.7 us, 6: 114.3, 4: 114.1, 3: 113.9, 2: 116.4 us). The
        // 8-bit variants, whose math warps run more code, take 2 (the
        // tensor-core E4M3 step 73.6 -> 70.9 us, the int8 step 89.9 -> 88.6 us).
        constexpr int LA = QK != 0 ? 2 : 4;
        constexpr int CPR = Cfg::ROWB / 16;          // 16-byte chunks per K/V row
        constexpr int CPRQ = Cfg::QROWB / 16;        // 16-byte chunks per q row
        const int pt = tid - Cfg::CW * 32;            // 0 .. kProducerThreads-1
        const int bpt = Cfg::TT / p.B;                // blocks per tile
        const int tpb = kProducerThreads / bpt;       // producer threads per block
        const int jblk = pt / tpb;
        const int tb = pt - jblk * tpb;
        const int jrow0 = jblk * p.B;                 // first tile row of this thread's block
        const uint8_t *kpool = static_cast<const uint8_t *>(p.kp);
        const uint8_t *vpool = FLAT ? kpool + p.v_off : static_cast<const uint8_t *>(p.vp);
        PkvCursor cur, la;
        pkv_cursor_at(cur, t_begin, seq_prefix, seq_len, W, Cfg::TT);
        la = cur;
        // prefix-aware: the cursors jump from section 0's range to section 1's
        int la_it = 0;
        auto advance = [&](PkvCursor &c, int next_it) {
            if (PFX && next_it == n0) cursor_jump(c, b1, seq_prefix, seq_len, W, Cfg::TT);
            else pkv_cursor_next(c, seq_len, W, p.U, Cfg::TT);
        };
        // per tile: the physical block of this thread's rows, or (flat
        // spans) the sequence's slot
        // 8-bit caches: the pools stream through L2 once per call, so their
        // lines are marked to go first (measured: the 8-bit decode 3 % faster;
        // the 16-bit step, which overlaps the next call's start with this
        // one's end, 0.7 % slower, so 16-bit copies keep the default policy)
        const uint64_t pol_stream = QK != 0 ? l2_policy_evict_first() : 0ull;
        // prefix-aware: a shared prefix is read by every chunk of its sharers'
        // heads, so its lines are kept (evict_last) and the rest stream by
        const uint64_t pol_keep = PFX ? l2_policy_evict_last() : 0ull;
        const uint64_t pol_pass = PFX ? l2_policy_evict_normal() : 0ull;
        auto load_entry = [&](const PkvCursor &c) -> int {
            const int ntok = min(Cfg::TT, c.L - c.ti * Cfg::TT);
            if (jblk * p.B >= ntok) return -1;
            if constexpr (FLAT) return __ldg(p.slots + c.s);
            if constexpr (PFX) return __ldg(p.block_tables + seq_tab[c.s] + c.ti * bpt + jblk);
            return __ldg(p.block_tables + (size_t)c.s * p.M + c.ti * bpt + jblk);
        };
        int ent[LA];
#pragma unroll
        for (int k = 0; k < LA; ++k) {
            ent[k] = -1;
            if (k < n_my) {
                ent[k] = load_entry(la);
                advance(la, ++la_it);
            }
        }
        // before the first q or pool byte; with pending_tail, q and the rows
        // below each sequence's last pending_tail are complete already and the
        // wait comes before the first tile holding one of those last rows
        if (!waited && p.pending_tail == 0) {
            grid_dependency_wait();
            waited = true;
        }
        // This thread's chunks sit at the same places in every tile: row of
        // the tile, swizzled shared-memory offset and byte offset inside the
        // (block, kv head) chunk of the pool, computed once.
        constexpr int NCH = Cfg::TT * CPR / kProducerThreads;   // K (and V) chunks per thread per tile
        int crow[NCH];
        uint32_t soff[NCH], goff[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int idx = tb + c * tpb;             // chunk within the block
            const int rb = idx / CPR, ch = idx - (idx / CPR) * CPR;
            crow[c] = jblk * p.B + rb;
            soff[c] = swz<Cfg::TT>(0u, crow[c], ch);
            // paged: row rb of a (block, kv head) chunk; flat: row crow of the
            // tile, Hk rows apart per token
            goff[c] = FLAT ? (uint32_t)(crow[c] * p.Hk * Cfg::ROWB + ch * 16)
                           : (uint32_t)(rb * Cfg::ROWB + ch * 16);
        }
        const size_t blk_stride = (size_t)p.Hk * p.B * Cfg::ROWB;   // bytes per pool block
        // unit values, refreshed at each segment's first tile
        int h0 = 0, gca = 0;
        size_t head_off = 0, head_rows = 0;
        // fused append (FUSED variants): the newest row of each context comes
        // from k_new / v_new, so the pool holds rows 0 .. L - 2 of it
        static_assert(!FUSED || (!FLAT && QK == 0), "the fused append is for paged 16/32-bit caches");
        const bool drop_first = p.drop_arrival && cta == 0 && pt == 0;   // test hook
        bool ok = true;
        for (int it0 = 0; it0 < n_my && ok; it0 += LA) {
#pragma unroll
            for (int k = 0; k < LA; ++k) {
                const int it = it0 + k;
                if (it >= n_my || !ok) break;
                const int e = ent[k];
                if (it + LA < n_my) {
                    ent[k] = load_entry(la);
                    advance(la, ++la_it);
                }
                const int stage = it % Cfg::NST;
                const uint32_t ph = (uint32_t)(it / Cfg::NST) & 1u;
                if (!mbar_wait(empty0 + 8 * stage, ph ^ 1u, p.err, p.wait_ns)) {
                    ok = false;
                    break;
                }
                const int ntok = min(Cfg::TT, cur.L - cur.ti * Cfg::TT);
                // fused append: tile row of the context's newest row (the last
                // row of the unit's last tile), -1 elsewhere
                const int rnew = (FUSED && cur.ti == cur.n - 1) ? ntok - 1 : -1;
                // pool rows of this tile end at pool_end; with pending_tail n the
                // last n rows of the context may still be written by the
                // preceding kernel (a fused append's newest row is not a pool row)
                const int pool_end = cur.ti * Cfg::TT + ntok - (FUSED && rnew >= 0 ? 1 : 0);
                if (!waited && pool_end > cur.L - p.pending_tail) {
                    grid_dependency_wait();   // the same tiles for every producer thread
                    waited = true;
                }
                const bool first = (it == 0) || (cur.ti == 0) || (PFX && it == n0);
                if (first) {
                    const int g = p.NC == 1 ? cur.u : cur.u / p.NC;
                    const int chunk = cur.u - g * p.NC;
                    h0 = g * p.G + chunk * p.GC;
                    gca = min(p.GC, p.G - chunk * p.GC);
                    if constexpr (PFX)   // a prefix unit: G heads of each of its members
                        if (cur.s < nv) gca = pm.w[cur.s].nm * p.G;

                    head_rows = (size_t)g * p.B;               // rows before kv head g in a block
                    head_off = FLAT ? (size_t)g * Cfg::ROWB : head_rows * Cfg::ROWB;
                }
                const uint32_t full = full0 + 8 * stage;
                const uint32_t sK = sbase + stage * Cfg::STAGE;
                const uint32_t sV = sK + Cfg::KVB;
                const uint32_t sS = sV + Cfg::KVB;           // scales (8-bit caches)
                const uint32_t sQ = sS + Cfg::SCB;
                // ---- K and V rows of block jblk of this tile
                const bool blk_ok = e >= 0 && e < p.NB;
                if (tb == 0 && jblk * p.B < ntok && !blk_ok) atomicOr(p.err, PKV_DEVERR_BLOCK_ID);
                size_t blk_base = 0;
                if (blk_ok) {
                    blk_base = FLAT ? (size_t)e * p.slot_stride +
                                          (size_t)cur.ti * Cfg::TT * p.Hk * Cfg::ROWB +
                                          head_off
                                    : (size_t)e * blk_stride + head_off;
                }
                uint64_t pol_tile = pol_stream;
                if constexpr (PFX) pol_tile = cur.s < nv ? pol_keep : pol_pass;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    const bool v = blk_ok && crow[c] < ntok;
                    const size_t off = v ? blk_base + goff[c] : 0;
                    if constexpr (QK != 0 || PFX) {
                        cp_async_16_hint(sK + soff[c], kpool + off, v, pol_tile);
                        cp_async_16_hint(sV + soff[c], vpool + off, v, pol_tile);
                    } else {
                        cp_async_16(sK + soff[c], kpool + off, v);
                        cp_async_16(sV + soff[c], vpool + off, v);
                    }
                }
                if constexpr (FUSED) {
                    // the unit's last tile: its newest row's K and V rows go from
                    // k_new / v_new to the stage's side slot (zeros for a bad
                    // block id, as the pool copy would give); the math warp
                    // holding that row puts them in place before its tile step.
                    // The pool copy above also fetched the row's slot: whatever
                    // it holds is overwritten.
                    // The threads of the row's block copy it (their blk_ok is
                    // that block's). Out of line: the issue loop is unrolled
                    // and its code size shows in the instruction fetch.
                    if (rnew >= jrow0 && rnew < jrow0 + p.B)
                        copy_new_row<Cfg::ROWB>(sQ + Cfg::QB, p.k_new, p.v_new,
                                                (size_t)cur.s * p.Hk +
                                                    (p.NC == 1 ? cur.u : cur.u / p.NC),
                                                tb, tpb, blk_ok);
                }
                if constexpr (QK != 0) {
                    // the block's B row scales, 4 rows per 16-byte copy; the
                    // bytes of rows past the context are zeroed, not read
                    if (tb < p.B / 4) {
                        const int row = jblk * p.B + 4 * tb;
                        const int nrow = blk_ok ? min(4, max(0, ntok - row)) : 0;
                        const size_t so =
                            blk_ok ? (size_t)e * p.Hk * p.B + head_rows + 4 * tb : 0;
                        cp_async_16_n(sS + row * 4, p.ks + so, 4u * nrow);
                        cp_async_16_n(sS + Cfg::TT * 4 + row * 4, p.vs + so, 4u * nrow);
                    }
                }
                // ---- q rows of the unit ride along with its first tile
                if (first) {
                    if (PFX && cur.s < nv) {   // a prefix unit: rows of several members
                        if constexpr (PFX)
                            copy_q_members<Cfg::QROWB>(sQ, p.q, members + pm.w[cur.s].m0, p.G,
                                                       p.Hq, h0, gca, pt);
                    } else {
                        const uint8_t *qsrc = static_cast<const uint8_t *>(p.q) +
                                              ((size_t)(cur.s - nv) * p.Hq + h0) * Cfg::QROWB;
                        for (int i = pt; i < gca * CPRQ; i += kProducerThreads)
                            cp_async_16(sQ + i * 16, qsrc + (size_t)i * 16, true);
                    }
                }
                // test hook (off unless a test asks for it): CTA 0's first
                // producer thread withholds its arrival on its first stage, so
                // the math warps' wait for that stage runs out
                if (!(drop_first && it == 0)) cp_async_arrive_noinc(full);
                if (pt == 0) {
                    const int64_t T_u = (int64_t)seq_prefix[cur.s] + (int64_t)cur.u * cur.n;
                    const bool last = (it == n_my - 1) || (cur.ti == cur.n - 1) ||
                                      (PFX && it == n0 - 1);
                    const bool sec0 = PFX && it < n0;   // the tile's section and its range here
                    const int64_t rb = sec0 ? b0 : b1, re = sec0 ? e0 : e1;
                    const bool whole = (T_u >= rb) && (T_u + cur.n <= re);
                    TileMeta mt;
                    mt.s = cur.s;
                    mt.h0 = h0;
                    mt.gca = gca;
                    mt.ntok = ntok;
                    mt.flags = (first ? kFirst : 0) | (last ? kLast : 0) | (whole ? kWhole : 0) |
                               (FUSED && rnew >= 0 ? kNewRow : 0);
                    mt.slot = (T_u > rb ? 1 : 0) + (PFX && !sec0 ? 2 : 0);
                    mt.tu = (int)T_u;
                    mt.nu = cur.n;
                    meta[stage] = mt;
                    mbar_arrive(full);   // release: the record is visible with the data
                }
                advance(cur, it + 1);
            }
        }
        if constexpr (FUSED) {
            if (ok) fused_append_rows<Cfg>(p, seq_prefix, seq_len, t_begin, e1, pt, waited);
        }
        cp_async_wait_all();   // this thread's copies land before it exits
        return;
    }

    // ======================= consumer warps =======================
    using Cs = typename std::conditional<Cfg::TC, TcConsumer<T, D, GMAX>,
                                         Consumer<T, D, GMAX, MMA, QK>>::type;
    Cs cs;
    // TC: warp 0 allocates TMEM (per group g: S at column 64g, O at 64g + 32)
    // and frees them once every math warp has arrived on the done barrier,
    // on every way out of the loop below
    uint32_t tmem_base = 0;
    const uint32_t tslot = tcx + Cfg::TCX_TSLOT;
    const uint32_t bar_tready = tcbar + 8 * (4 * Cfg::NG), bar_done = bar_tready + 8;
    auto tc_leave = [&]() {
        if constexpr (Cfg::TC) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_done);
            if (warp == 0) {
                mbar_wait(bar_done, 0, p.err, 4 * p.wait_ns);
                tc_fence_after();
                __syncwarp();
                tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
            }
        }
    };
    if constexpr (Cfg::TC) {
        __syncwarp();
        if (warp == 0) {
            tmem_alloc(tslot, Cfg::TMEM_COLS);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tready);
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_tready, 0, p.err, p.wait_ns));
        tc_fence_after();
        tmem_base = ok || warp == 0 ? lds_u32(tslot) : 0u;
        if (!ok) {
            tc_leave();
            return;
        }
        const uint32_t tb = tcbar;
        cs.g = warp >> 2;
        cs.qw = warp & 3;
        cs.r = cs.qw * 32 + lane;
        cs.issuer = cs.qw == 0;
        cs.tS = tmem_base + ((uint32_t)(cs.qw * 32) << 16) + 64 * cs.g;
        cs.tO = cs.tS + 32;
        cs.qp = sbase + Cfg::OFF_TC + Cfg::TCG * cs.g;
        cs.pb = cs.qp + Cfg::TCG / 2;
        cs.xbuf = tcx + 8 * Cfg::XS * cs.g;
        cs.qsc = tcx + Cfg::TCX_QSC + 32 * cs.g;
        cs.barS = tb + 8 * (0 * Cfg::NG + cs.g);
        cs.barO = tb + 8 * (1 * Cfg::NG + cs.g);
        cs.barX = tb + 8 * (2 * Cfg::NG + cs.g);
        cs.barP = tb + 8 * (3 * Cfg::NG + cs.g);
        cs.err = p.err;
        cs.wait_ns = p.wait_ns;
    } else if constexpr (MMA) {
        cs.pbuf = sbase + Cfg::OFF_PBUF + warp * Cfg::NTN * 512;
    }
    cs.reset();
    int seg = 0;
    // Cut segments whose partial this warp has written (a range's first and
    // last segment at most, per section). Counting them waits until the CTA's tiles are
    // done: the fence that must come before a count would otherwise wait
    // behind the copies in flight and stall the math warps mid-run.
    PendSegT<PFX> pend[SLOTS];   // two per section of the work list
    int n_pend = 0;
    // prefix-aware: (sequence, kv head) entries whose result slices this warp
    // has written, counted at the CTA's end like the cut segments
    int *fin_list = reinterpret_cast<int *>(smem + Cfg::OFF_FIN) + warp * kFinCap;
    int n_fin = 0;
    for (int it = 0; it < n_my; ++it) {
        const int stage = it % Cfg::NST;
        const uint32_t ph = (uint32_t)(it / Cfg::NST) & 1u;
        bool full_ok = mbar_wait(full0 + 8 * stage, ph, p.err, p.wait_ns);
        if constexpr (Cfg::TC) full_ok = __all_sync(0xffffffffu, full_ok);
        if (!full_ok) {
            tc_leave();
            return;
        }
        const TileMeta mt = meta[stage];
        const uint32_t sK = sbase + stage * Cfg::STAGE;
        const uint32_t sV = sK + Cfg::KVB;
        if (mt.flags & kFirst) {
            if constexpr (Cfg::TC) {
                if (!cs.first(smem + stage * Cfg::STAGE + 2 * Cfg::KVB + Cfg::SCB, mt.gca,
                              p.scale_log2, lane)) {
                    tc_leave();
                    return;
                }
            } else {
                cs.reset();
                cs.load_q(smem + stage * Cfg::STAGE + 2 * Cfg::KVB + Cfg::SCB, mt.gca,
                          p.scale_log2, lane);
            }
        }
        if constexpr (FUSED) {
            // the context's newest row: the math warp whose 16 rows hold it
            // copies its K and V rows from the side slot into the tile (no
            // other warp reads those rows)
            if ((mt.flags & kNewRow) && (mt.ntok - 1) / 16 == warp) {
                constexpr int CPRw = Cfg::ROWB / 16;
                const int rn = mt.ntok - 1;
                const uint32_t side = sK + 2 * Cfg::KVB + Cfg::SCB + Cfg::QB;
#pragma unroll
                for (int i = lane; i < 2 * CPRw; i += 32) {
                    uint32_t a, b, c2, d;
                    lds_u32x4(side + i * 16, a, b, c2, d);
                    const uint32_t dst = i < CPRw ? swz<Cfg::TT>(sK, rn, i)
                                                  : swz<Cfg::TT>(sV, rn, i - CPRw);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(a),
                                 "r"(b), "r"(c2), "r"(d)
                                 : "memory");
                }
                __syncwarp();
            }
        }
        if constexpr (Cfg::TC) {
            // the group whose turn it is runs the tile's products on the tensor cores
            const uint32_t ksc = sK + 2 * Cfg::KVB;
            if (it % Cfg::NG == cs.g && !cs.tile(sK, sV, ksc, ksc + 4 * Cfg::TT, mt.ntok, lane)) {
                tc_leave();
                return;
            }
        } else if constexpr (QK != 0) {
            // the tile step reads this warp's 16 rows of codes straight into registers
            const uint32_t ksc = sK + 2 * Cfg::KVB;
            cs.tile(sK, sV, mt.ntok, warp, lane, ksc, ksc + 4 * Cfg::TT);
        } else {
            cs.tile(sK, sV, mt.ntok, warp, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);

        if (mt.flags & kLast) {
            // combine the math warps' softmax states for this segment. Merge
            // slice `slice` < kMergeSlices owns the outputs idx = slice*32 +
            // lane + 128k: warp `slice` (TC: warp slice of the group that ran
            // the segment's last tile, while the other groups go on; they
            // only feed the combine)
            int slice = warp;
            if constexpr (Cfg::TC) slice = it % Cfg::NG == cs.g ? cs.qw : kMergeSlices;
            if (!mbar_wait(comb_empty, ((uint32_t)seg & 1u) ^ 1u, p.err, p.wait_ns)) {
                tc_leave();
                return;
            }
            cs.write_comb(comb_o, comb_m, comb_l, warp, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(comb_full);
            if (Cfg::TC && slice >= kMergeSlices) {
                ++seg;
                continue;
            }
            if (!mbar_wait(comb_full, (uint32_t)seg & 1u, p.err, p.wait_ns)) {
                tc_leave();
                return;
            }
            if (!waited && slice < kMergeSlices) {   // stores wait for the preceding kernel
                grid_dependency_wait();
                waited = true;
            }
            const int base = (cta * SLOTS + mt.slot) * p.GC;
            const bool whole = (mt.flags & kWhole) != 0;
            UnitDest ud{0, mt.s, 0};
            if constexpr (PFX) {
                if (mt.s < nv) ud = UnitDest{1, 0, pm.w[mt.s].m0};
                else ud = UnitDest{pm.w[mt.s].blocks > 0 ? 2 : 0, mt.s - nv, 0};
            }
            // slice `slice` < kMergeSlices owns the elements idx = slice*32 +
            // lane + 128k of the unit's gca x D outputs (head j = idx / D,
            // element d = idx % D)
            if constexpr (Cfg::TC) {
                // warp groups: m and O per group, l in shares per warp
                if (slice < kMergeSlices) {
                    const int d = slice * 32 + lane;
#pragma unroll
                    for (int k = 0; k < GMAX; ++k) {
                        if (k >= mt.gca) break;
                        float M = -CUDART_INF_F;
#pragma unroll
                        for (int gi = 0; gi < Cfg::NG; ++gi) M = fmaxf(M, comb_m[4 * gi * GMAX + k]);
                        float Ls = 0.f, O = 0.f;
#pragma unroll
                        for (int gi = 0; gi < Cfg::NG; ++gi) {
                            const float w = exp2f(comb_m[4 * gi * GMAX + k] - M);
#pragma unroll
                            for (int q = 0; q < 4; ++q) Ls = fmaf(w, comb_l[(4 * gi + q) * GMAX + k], Ls);
                            O = fmaf(w, comb_o[(gi * GMAX + k) * D + d], O);
                        }
                        O /= Ls;
                        const float lse = M + log2f(Ls);
                        if (whole) {
                            store_out(p.out, ((size_t)mt.s * p.Hq + mt.h0 + k) * D + d,
                                      p.out_dtype, O);
                            if (p.lse_out && d == 0)
                                p.lse_out[(size_t)mt.s * p.Hq + mt.h0 + k] = lse;
                        } else {
                            p.ws_o[(size_t)(base + k) * D + d] = O;
                            if (lane == 0)
                                p.ws_lse[((cta * SLOTS + mt.slot) * kMergeSlices + slice) * p.GC + k] =
                                    lse;
                        }
                    }
                }
            } else if constexpr (MMA && D == 128) {
                // Weights first: lane L holds the (warp w, head j) pairs P = 32s + L
                // (P = w * GMAX + j), reduces max and sum over w with shuffles and
                // keeps w's weight 2^(m_wj - M_j) / sum_w' 2^(m_w'j - M_j) l_w'j.
                // Element k of this lane (idx = warp*32 + lane + 128k) is head k,
                // d = warp*32 + lane; it needs only the CW weights of head k.
                constexpr int NPAIR = Cfg::CW * GMAX;
                constexpr int PPL = (NPAIR + 31) / 32;
                static_assert(NPAIR % 32 == 0 || NPAIR < 32, "pairs fill whole warps");
                if (slice < kMergeSlices) {
                    float mv[PPL], lv[PPL], sw[PPL];
                    float M = -CUDART_INF_F;
#pragma unroll
                    for (int q = 0; q < PPL; ++q) {
                        const int P = (32 * q + lane) % NPAIR;
                        mv[q] = comb_m[P];
                        lv[q] = comb_l[P];
                        M = fmaxf(M, mv[q]);
                    }
#pragma unroll
                    for (int o = GMAX; o < 32 && o < NPAIR; o <<= 1)
                        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                    float Lsum = 0.f;
#pragma unroll
                    for (int q = 0; q < PPL; ++q) {
                        sw[q] = exp2f(mv[q] - M);
                        Lsum = fmaf(sw[q], lv[q], Lsum);
                    }
#pragma unroll
                    for (int o = GMAX; o < 32 && o < NPAIR; o <<= 1)
                        Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
                    const float inv = 1.f / Lsum;
#pragma unroll
                    for (int q = 0; q < PPL; ++q) sw[q] *= inv;
                    const float lse_j = M + log2f(Lsum);   // head lane % GMAX
                    const int d = slice * 32 + lane;
#pragma unroll
                    for (int k = 0; k < GMAX; ++k) {
                        if (k >= mt.gca) break;
                        float O = 0.f;
#pragma unroll
                        for (int w = 0; w < Cfg::CW; ++w) {
                            const int P = w * GMAX + k;
                            const float wk = __shfl_sync(0xffffffffu, sw[P >> 5], P & 31);
                            O = fmaf(wk, comb_o[(w * GMAX + k) * D + comb_col<MMA, QK>(k, d)], O);
                        }
                        const float lse = __shfl_sync(0xffffffffu, lse_j, k);
                        if (whole) {
                            if constexpr (PFX) {
                                put_result<D>(p, ud, mt.h0, k, d, O, lse, members, seq_len, nv);
                            } else {
                                store_out(p.out, ((size_t)mt.s * p.Hq + mt.h0 + k) * D + d,
                                          p.out_dtype, O);
                                if (p.lse_out && d == 0)
                                    p.lse_out[(size_t)mt.s * p.Hq + mt.h0 + k] = lse;
                            }
                        } else {
                            p.ws_o[(size_t)(base + k) * D + d] = O;
                            // lane 0 holds one element of every head in the slice:
                            // it writes the slice's copy of the head's lse
                            if (lane == 0)
                                p.ws_lse[((cta * SLOTS + mt.slot) * kMergeSlices + slice) * p.GC + k] =
                                    lse;
                        }
                    }
                }
            } else {
                const int idx0 = slice < kMergeSlices ? slice * 32 + lane : mt.gca * D;
                for (int idx = idx0; idx < mt.gca * D; idx += kMergeSlices * 32) {
                    const int j = idx / D, d = idx - (idx / D) * D;
                    float M = -CUDART_INF_F;
    #pragma unroll
                    for (int w = 0; w < Cfg::CW; ++w) M = fmaxf(M, comb_m[w * GMAX + j]);
                    float Ls = 0.f, O = 0.f;
    #pragma unroll
                    for (int w = 0; w < Cfg::CW; ++w) {
                        const float wt = exp2f(comb_m[w * GMAX + j] - M);
                        Ls = fmaf(wt, comb_l[w * GMAX + j], Ls);
                        O = fmaf(wt, comb_o[(w * GMAX + j) * D + comb_col<MMA, QK>(j, d)], O);
                    }
                    const float o = O / Ls;
                    if (whole) {
                        if constexpr (PFX) {
                            put_result<D>(p, ud, mt.h0, j, d, o, M + log2f(Ls), members, seq_len,
                                          nv);
                        } else {
                            store_out(p.out, ((size_t)mt.s * p.Hq + mt.h0 + j) * D + d,
                                      p.out_dtype, o);
                            if (p.lse_out && d == 0)
                                p.lse_out[(size_t)mt.s * p.Hq + mt.h0 + j] = M + log2f(Ls);
                        }
                    } else {
                        p.ws_o[(size_t)(base + j) * D + d] = o;
                        // lane 0 holds one element of every head in the slice:
                        // it writes the slice's copy of the head's lse
                        if (lane == 0)
                            p.ws_lse[((cta * SLOTS + mt.slot) * kMergeSlices + slice) * p.GC + j] =
                                M + log2f(Ls);
                    }
                }
            }
            if (!whole && slice < kMergeSlices && slice * 32 < mt.gca * D) {
                if constexpr (PFX) pend[n_pend++] = pend_seg_pfx(mt, C, NT0, NT, ud);
                else pend[n_pend++] = pend_seg(mt, C, NT);
            }
            if constexpr (PFX)
                if (whole && slice < kMergeSlices && ud.kind != 0)
                    note_final<D>(p, ud, mt.h0, mt.gca, members, seq_len, nv, fin_list, n_fin,
                                  warp, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(comb_empty);
            ++seg;
        }
    }
    tc_leave();
    // this warp's merge slice (TC: its place in its group)
    int mslice = warp;
    if constexpr (Cfg::TC) mslice = cs.qw;
    if (n_pend == 0) {
        if constexpr (PFX)
            if (n_fin) flush_final<D>(p, fin_list, n_fin, warp, lane);
        return;
    }
    // Count this warp's slices of its cut segments; for each unit, the last of
    // its partials to arrive merges the slice. Lane 0 releases the whole
    // warp's stores (ordered before it by __syncwarp) with its counts and
    // acquires the other partials with them.
    __syncwarp();
    unsigned prev[SLOTS] = {};
    if (lane == 0) {
        fence_acq_rel_gpu();
        for (int i = 0; i < n_pend; ++i) {
            int sec = 0;
            if constexpr (PFX) sec = pend[i].sec;
            prev[i] = atomicAdd(p.ws_cnt + (pend[i].c_first + sec * C) * kMergeSlices + mslice, 1u);
        }
        fence_acq_rel_gpu();
    }
    __syncwarp();
    for (int i = 0; i < n_pend; ++i) {
        const PendSegT<PFX> &ps = pend[i];
        if ((int)__shfl_sync(0xffffffffu, prev[i], 0) + 1 == ps.parts) {
            int sec = 0;
            if constexpr (PFX) sec = ps.sec;
            if (lane == 0)   // for the next call
                p.ws_cnt[(ps.c_first + sec * C) * kMergeSlices + mslice] = 0u;
            merge_slice<D, GMAX, SLOTS, PFX>(p, ps, mslice, lane, NT, members, seq_len, nv);
            if constexpr (PFX)
                if (ps.ud.kind != 0)
                    note_final<D>(p, ps.ud, ps.mt.h0, ps.mt.gca, members, seq_len, nv, fin_list,
                                  n_fin, warp, lane);
        }
    }
    if constexpr (PFX)
        if (n_fin) flush_final<D>(p, fin_list, n_fin, warp, lane);
}

// ---------------------------------------------------------------------------
// host-side launch of one variant
// ---------------------------------------------------------------------------
template <typename T, int D, int GMAX, bool MMA, int QK = 0, bool FLAT = false, bool FUSED = false,
          bool PFX = false>
struct SplitVariant {
    using Cfg = SplitCfg<T, D, GMAX, MMA, QK, FUSED, PFX>;
    using PM = typename std::conditional<PFX, PrefixMap, NoPrefixMap>::type;

    static constexpr auto kernel() { return decode_split_kernel<T, D, GMAX, MMA, QK, FLAT, FUSED, PFX>; }

    // Per-device state lives in atomics: host threads making their first
    // calls on a device at the same time may both set the attribute (the
    // same value, so harmless), but never read a half-written flag.
    static cudaError_t prepare(int dev) {
        static std::atomic<bool> done[64];
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!done[dev].load(std::memory_order_acquire)) {
            const size_t smem = Cfg::smem_bytes(kMaxSeqsPerLaunch);
            cudaError_t e = cudaFuncSetAttribute(kernel(),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            done[dev].store(true, std::memory_order_release);
        }
        return cudaSuccess;
    }

    // W work sequences: the batch, plus the virtual prefix ones (prefix-aware)
    static cudaError_t launch_with(const DecodeParams &p, const PM &pm, int W, cudaStream_t st) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = prepare(dev);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)p.C);
        cfg.blockDim = dim3(Cfg::THREADS);
        cfg.dynamicSmemBytes = Cfg::smem_bytes(W);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel(), p, pm);
    }

    static cudaError_t launch(const DecodeParams &p, cudaStream_t st) {
        if constexpr (PFX) return cudaErrorInvalidValue;   // needs the prefix map
        else return launch_with(p, PM{}, p.S, st);
    }

    static cudaError_t launch_prefix(const DecodeParams &p, const PrefixMap &pm, cudaStream_t st) {
        if constexpr (PFX) return launch_with(p, pm, pm.nv + p.S, st);
        else return cudaErrorInvalidValue;
    }

    // occupancy of this variant on the current device (queried once per device)
    static int max_ctas_per_sm() {
        static std::atomic<int> cached[64];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
        const int c = cached[dev].load(std::memory_order_acquire);
        if (c > 0) return c;
        if (prepare(dev) != cudaSuccess) return 0;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel(), Cfg::THREADS,
                                                          Cfg::smem_bytes(kMaxSeqsPerLaunch)) !=
            cudaSuccess)
            return 0;
        cached[dev].store(n, std::memory_order_release);
        return n;
    }

    static const DecodeVariant *get() {
        static const DecodeVariant v{PFX ? nullptr : &launch, &max_ctas_per_sm,
                                     PFX ? &launch_prefix : nullptr};
        return &v;
    }
};

}  // namespace pkv
