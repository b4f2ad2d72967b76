// Prefix-aware decode: sequences that share their leading blocks read those
// blocks once per group of sharers (include/pkv.h, pkv_decode_attention_prefix).
//
// Passage: identical prompt prefixes are stored once and shared by every
// request that holds them ("KV-Cache Optimization & PagedAttention for
// Long-Context Agents", section "Key KV-Cache Optimization Principles", item
// 3; "PagedAttention — Math + Memory Model", section "Copy-on-write: sharing
// blocks across samples"). Reading them once per group instead of once per
// sequence is this library's use of that sharing.
//
// Attention over a context split into a shared prefix P and a private suffix
// S is the log-sum-exp merge of the two partial attentions:
//     out = (2^{l_P} o_P + 2^{l_S} o_S) / (2^{l_P} + 2^{l_S}),
// l_X = log2 sum_{t in X} exp(scaled score), o_X the attention over X alone.
// The library computes o_P for all sharers at once: their q heads are
// gathered under each kv head and cut into virtual sequences of
// kPrefixHeads heads per kv head, all over the prefix, so a prefix block
// feeds that many sharers' heads per pass of the decode kernel (the 8-head
// variant, whose code the suffix decode also runs). o_S is an ordinary
// decode over each sequence's table shifted past its prefix. A last kernel
// merges.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <vector>

#include "../../include/pkv.h"
#include "device_utils.cuh"
#include "pkv_internal.h"

namespace {

// rows of q (D elements) gathered by index: dst row r = src row idx[r]
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4 *__restrict__ src,
                                                          uint4 *__restrict__ dst,
                                                          const int32_t *__restrict__ idx,
                                                          int rows, int vec_per_row) {
    const int64_t total = (int64_t)rows * vec_per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / vec_per_row), v = (int)(i - (int64_t)r * vec_per_row);
        dst[i] = __ldg(src + (size_t)__ldg(idx + r) * vec_per_row + v);
    }
}

// Suffix tables and lengths: table row s shifted left by shift[s] entries.
// Then the prefix tables of the virtual sequences: row r (Mp entries) holds
// the first vpb[r] entries of table row vsrc[r] (a member of the group).
__global__ void __launch_bounds__(256) suffix_tables_kernel(
    const int32_t *__restrict__ tables, const int32_t *__restrict__ lens,
    const int32_t *__restrict__ shift, int S, int M, int B, int32_t *__restrict__ suf_tables,
    int32_t *__restrict__ suf_lens, const int32_t *__restrict__ vsrc,
    const int32_t *__restrict__ vpb, int NV, int Mp, int32_t *__restrict__ vtab, unsigned *err) {
    const int64_t nsuf = (int64_t)S * M;
    const int64_t total = nsuf + (int64_t)NV * Mp;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        if (i < nsuf) {
            const int s = (int)(i / M), j = (int)(i - (int64_t)s * M);
            const int sh = __ldg(shift + s);
            suf_tables[i] = j + sh < M ? __ldg(tables + (size_t)s * M + j + sh) : -1;
            if (j == 0) {
                const int rest = __ldg(lens + s) - sh * B;
                if (rest < 0) atomicOr(err, PKV_DEVERR_CONTEXT);
                suf_lens[s] = rest < 0 ? 0 : rest;
            }
        } else {
            const int64_t k = i - nsuf;
            const int r = (int)(k / Mp), j = (int)(k - (int64_t)r * Mp);
            vtab[k] = j < __ldg(vpb + r) ? __ldg(tables + (size_t)__ldg(vsrc + r) * M + j) : 0;
        }
    }
}

// out[s][h] = log-sum-exp merge of the prefix part (row pref_row[s*Hq+h] of
// o_pref, or none when -1) and the suffix part
__global__ void __launch_bounds__(256) merge_prefix_kernel(
    const float *__restrict__ o_pref, const float *__restrict__ lse_pref,
    const int32_t *__restrict__ pref_row, const float *__restrict__ o_suf,
    const float *__restrict__ lse_suf, int rows, int D, void *out, int out_dtype) {
    const int64_t total = (int64_t)rows * D;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / D), d = (int)(i - (int64_t)r * D);
        const int pr = __ldg(pref_row + r);
        const float lp = pr >= 0 ? __ldg(lse_pref + pr) : -CUDART_INF_F;
        const float ls = __ldg(lse_suf + r);
        const float m = fmaxf(lp, ls);
        float v = 0.f;
        if (m > -CUDART_INF_F) {
            const float wp = exp2f(lp - m), ws = exp2f(ls - m);
            const float op = pr >= 0 ? __ldg(o_pref + (size_t)pr * D + d) : 0.f;
            v = (wp * op + ws * __ldg(o_suf + i)) / (wp + ws);
        }
        pkv::store_out(out, (size_t)i, out_dtype, v);
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// q heads per kv head of one virtual prefix sequence
constexpr int kPrefixHeads = 8;

// Sizes and host-side index arrays of one prefix-aware call.
struct PrefixPlan {
    int S, Hq, Hk, Gq, M, B, D, G;
    std::vector<std::vector<int32_t>> members;   // per group
    std::vector<int32_t> qidx;                   // gathered q row -> source row
    std::vector<int32_t> pref_row;               // [S*Hq] row of o_pref, or -1
    std::vector<int32_t> shift;                  // [S] leading blocks to skip
    std::vector<size_t> group_row0;              // first gathered row of each group
    std::vector<int> group_v0, group_nv;         // first virtual sequence, their number
    std::vector<int32_t> vsrc, vpb, vlen;        // per virtual sequence: table row, blocks, tokens
    int total_rows = 0, NV = 0, Mp = 1;
    size_t split_ws = 0, off_q = 0, off_op = 0, off_lp = 0, off_os = 0, off_ls = 0, off_tab = 0,
           off_vtab = 0, off_len = 0, off_idx = 0, bytes = 0;
};

pkv_status plan_prefix(const pkv_cache_desc *c, int32_t S, int32_t Hq, int32_t M,
                       const pkv_prefix_groups *g, int32_t num_ctas, PrefixPlan *pp) {
    if (!c || !g) return pkv::set_last_error(PKV_ERR_INVALID_ARG, "NULL argument");
    if (S < 0 || M < 1 || Hq < 1 || Hq % c->num_kv_heads != 0)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "bad sizes");
    if (g->num_groups < 0 || (S > 0 && !g->group_of_seq) ||
        (g->num_groups > 0 && !g->group_prefix_blocks))
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "bad prefix groups");
    PrefixPlan &p = *pp;
    p.S = S;
    p.Hq = Hq;
    p.Hk = c->num_kv_heads;
    p.Gq = Hq / p.Hk;
    p.M = M;
    p.B = c->block_size;
    p.D = c->head_dim;
    p.G = g->num_groups;
    p.members.assign(p.G, {});
    p.shift.assign(S, 0);
    for (int32_t s = 0; s < S; ++s) {
        const int32_t gi = g->group_of_seq[s];
        if (gi < -1 || gi >= p.G)
            return pkv::set_last_error(PKV_ERR_INVALID_ARG, "group_of_seq[%d] = %d", s, gi);
        if (gi >= 0) p.members[gi].push_back(s);
    }
    p.group_row0.resize(p.G);
    p.group_v0.resize(p.G);
    p.group_nv.resize(p.G);
    p.pref_row.assign((size_t)S * Hq, -1);
    constexpr int KH = kPrefixHeads;
    for (int32_t gi = 0; gi < p.G; ++gi) {
        const int32_t pb = g->group_prefix_blocks[gi];
        if (pb < 1 || pb > M || p.members[gi].empty())
            return pkv::set_last_error(PKV_ERR_INVALID_ARG,
                                       "group %d: prefix of %d blocks, %zu members", gi, pb,
                                       p.members[gi].size());
        const int J = (int)p.members[gi].size();
        // The J*Gq heads under each kv head, m = j*Gq + i, go to virtual
        // sequence m / KH, head (kh, m % KH): gathered row
        // row0 + (v*Hk + kh)*KH + m % KH. Rows past J*Gq repeat a real
        // head; their outputs are not read.
        const int nv = (J * p.Gq + KH - 1) / KH;
        p.group_row0[gi] = p.total_rows;
        p.group_v0[gi] = p.NV;
        p.group_nv[gi] = nv;
        for (int v = 0; v < nv; ++v)
            for (int kh = 0; kh < p.Hk; ++kh)
                for (int i8 = 0; i8 < KH; ++i8) {
                    const int m = v * KH + i8;
                    const int mm = m < J * p.Gq ? m : 0;
                    const int s = p.members[gi][mm / p.Gq], h = kh * p.Gq + mm % p.Gq;
                    const int r = p.total_rows + (v * p.Hk + kh) * KH + i8;
                    p.qidx.push_back(s * Hq + h);
                    if (m < J * p.Gq) p.pref_row[(size_t)s * Hq + h] = r;
                }
        for (int v = 0; v < nv; ++v) {
            p.vsrc.push_back(p.members[gi][0]);
            p.vpb.push_back(pb);
            p.vlen.push_back(pb * p.B);
        }
        if (pb > p.Mp) p.Mp = pb;
        for (int s : p.members[gi]) p.shift[s] = pb;
        p.total_rows += nv * p.Hk * KH;
        p.NV += nv;
    }
    // the split-K workspace serves every decode of the call (they run in
    // stream order); it leads, so a zero-filled workspace keeps its counters
    const size_t w1 = pkv_decode_workspace_bytes_ex(c, Hq, num_ctas);
    const size_t w2 = p.G ? pkv_decode_workspace_bytes_ex(c, p.Hk * KH, num_ctas) : 0;
    if (w1 == 0 || (p.G && w2 == 0))
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "split-K workspace query failed");
    const size_t es = c->dtype == PKV_F32 ? 4 : 2;
    p.split_ws = align256(w1 > w2 ? w1 : w2);
    p.off_q = p.split_ws;
    p.off_op = p.off_q + align256((size_t)p.total_rows * p.D * es);
    p.off_lp = p.off_op + align256((size_t)p.total_rows * p.D * 4);
    p.off_os = p.off_lp + align256((size_t)p.total_rows * 4);
    p.off_ls = p.off_os + align256((size_t)S * Hq * p.D * 4);
    p.off_tab = p.off_ls + align256((size_t)S * Hq * 4);
    p.off_vtab = p.off_tab + align256((size_t)S * M * 4);
    p.off_len = p.off_vtab + align256((size_t)p.NV * p.Mp * 4);
    p.off_idx = p.off_len + align256((size_t)S * 4);
    p.bytes = p.off_idx +
              align256((p.qidx.size() + p.pref_row.size() + S + 3 * (size_t)p.NV) * 4);
    return PKV_OK;
}

int grid_for(int64_t n) {
    int64_t b = (n + 255) / 256;
    return (int)(b < 1 ? 1 : (b > 4096 ? 4096 : b));
}

}  // namespace

extern "C" {

size_t pkv_decode_prefix_workspace_bytes(const pkv_cache_desc *cache, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_blocks_per_seq,
                                         const pkv_prefix_groups *groups, int32_t num_ctas) {
    PrefixPlan pp;
    if (plan_prefix(cache, num_seqs, num_q_heads, max_blocks_per_seq, groups, num_ctas, &pp) !=
        PKV_OK)
        return 0;
    return pp.bytes;
}

pkv_status pkv_decode_attention_prefix(const pkv_cache_desc *cache, const void *q,
                                       int32_t num_seqs, int32_t num_q_heads, const void *k_pool,
                                       const void *v_pool, const int32_t *block_tables,
                                       int32_t max_blocks_per_seq, const int32_t *context_lens,
                                       float scale, const pkv_prefix_groups *groups, void *out,
                                       int32_t out_dtype, void *workspace,
                                       size_t workspace_bytes, void *stream,
                                       const pkv_decode_options *options) {
    const int32_t num_ctas = options ? options->num_ctas : 0;
    PrefixPlan pp;
    pkv_status st = plan_prefix(cache, num_seqs, num_q_heads, max_blocks_per_seq, groups,
                                num_ctas, &pp);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !block_tables || !context_lens || !out || !k_pool || !v_pool)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "a pointer argument is NULL");
    if (out_dtype != PKV_F32 && out_dtype != PKV_F16 && out_dtype != PKV_BF16)
        return pkv::set_last_error(PKV_ERR_UNSUPPORTED, "out_dtype %d", out_dtype);
    if (!workspace || workspace_bytes < pp.bytes)
        return pkv::set_last_error(PKV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given",
                                   pp.bytes, workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(workspace)) % 16)
        return pkv::set_last_error(PKV_ERR_INVALID_ARG, "q and the workspace must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t es = cache->dtype == PKV_F32 ? 4 : 2;
    const int S = num_seqs, Hq = num_q_heads, D = pp.D, M = max_blocks_per_seq;
    int32_t *d_len = reinterpret_cast<int32_t *>(ws + pp.off_len);      // [S] suffix tokens
    int32_t *d_idx = reinterpret_cast<int32_t *>(ws + pp.off_idx);
    int32_t *d_qidx = d_idx;
    int32_t *d_pref_row = d_qidx + pp.qidx.size();
    int32_t *d_shift = d_pref_row + pp.pref_row.size();
    int32_t *d_vsrc = d_shift + S;           // per virtual prefix sequence
    int32_t *d_vpb = d_vsrc + pp.NV;
    int32_t *d_vlen = d_vpb + pp.NV;
    // index arrays and the virtual sequences' tables and lengths: staged
    // from the host in one copy
    std::vector<int32_t> stage(pp.qidx);
    stage.insert(stage.end(), pp.pref_row.begin(), pp.pref_row.end());
    stage.insert(stage.end(), pp.shift.begin(), pp.shift.end());
    stage.insert(stage.end(), pp.vsrc.begin(), pp.vsrc.end());
    stage.insert(stage.end(), pp.vpb.begin(), pp.vpb.end());
    stage.insert(stage.end(), pp.vlen.begin(), pp.vlen.end());
    cudaError_t e = cudaMemcpyAsync(d_idx, stage.data(), stage.size() * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess)
        return pkv::set_last_error(PKV_ERR_CUDA, "staging: %s", cudaGetErrorString(e));
    unsigned *err = nullptr;
    if ((st = pkv::device_error_word(&err)) != PKV_OK) return st;
    // gathered q for the prefixes; suffix tables and lengths
    uint8_t *d_q = ws + pp.off_q;
    const int vpr = (int)(D * es / 16);
    if (pp.total_rows)
        gather_rows_kernel<<<grid_for((int64_t)pp.total_rows * vpr), 256, 0, s>>>(
            static_cast<const uint4 *>(q), reinterpret_cast<uint4 *>(d_q), d_qidx, pp.total_rows,
            vpr);
    int32_t *d_tab = reinterpret_cast<int32_t *>(ws + pp.off_tab);
    int32_t *d_vtab = reinterpret_cast<int32_t *>(ws + pp.off_vtab);
    suffix_tables_kernel<<<grid_for((int64_t)S * M + (int64_t)pp.NV * pp.Mp), 256, 0, s>>>(
        block_tables, context_lens, d_shift, S, M, pp.B, d_tab, d_len, d_vsrc, d_vpb, pp.NV, pp.Mp,
        d_vtab, err);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return pkv::set_last_error(PKV_ERR_CUDA, "prefix set-up launch: %s", cudaGetErrorString(e));
    float *o_pref = reinterpret_cast<float *>(ws + pp.off_op);
    float *l_pref = reinterpret_cast<float *>(ws + pp.off_lp);
    float *o_suf = reinterpret_cast<float *>(ws + pp.off_os);
    float *l_suf = reinterpret_cast<float *>(ws + pp.off_ls);
    pkv_decode_options o = {};
    o.num_ctas = num_ctas;
    o.consumer = options ? options->consumer : 0;
    // each group's prefix, once per kPrefixHeads of its sharers' heads
    for (int gi = 0; gi < pp.G; ++gi) {
        const size_t r0 = pp.group_row0[gi];
        const int v0 = pp.group_v0[gi];
        o.lse_out = l_pref + r0;
        st = pkv_decode_attention_ex(cache, d_q + r0 * D * es, pp.group_nv[gi],
                                     pp.Hk * kPrefixHeads, k_pool, v_pool,
                                     d_vtab + (size_t)v0 * pp.Mp, pp.Mp, d_vlen + v0, scale,
                                     o_pref + r0 * D, PKV_F32, ws, pp.split_ws, stream, &o);
        if (st != PKV_OK) return st;
    }
    // every sequence's private suffix
    o.lse_out = l_suf;
    st = pkv_decode_attention_ex(cache, q, S, Hq, k_pool, v_pool, d_tab, M, d_len, scale, o_suf,
                                 PKV_F32, ws, pp.split_ws, stream, &o);
    if (st != PKV_OK) return st;
    merge_prefix_kernel<<<grid_for((int64_t)S * Hq * D), 256, 0, s>>>(
        o_pref, l_pref, d_pref_row, o_suf, l_suf, S * Hq, D, out, out_dtype);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return pkv::set_last_error(PKV_ERR_CUDA, "prefix merge launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // extern "C"
