"""Parity of the 8-bit KV cache path (pkv_append_quant, pkv_decode_attention_quant,
pkv_block_copy_quant) against the CPU oracle.

Each side quantizes the same drawn activations itself: the oracle in C on
the CPU, the library through pkv_append_quant on the GPU. Codes and scales
must then match bit for bit (both take the rounding decisions in fp32), and
the decode over the two caches must match within max-abs 2e-3.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_cache_47_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu

TOL = 2e-3
KINDS = ["int8", "fp8_e4m3"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()
    yield


def _empty_pools(NB, Hk, B, D, device):
    """Code pools full of 0x7F (E4M3 NaN, int8 127) and NaN scales: entries no
    append writes must never reach an output."""
    kc = torch.full((NB, Hk, B, D), 0x7F, dtype=torch.uint8, device=device)
    ks = torch.full((NB, Hk, B), float("nan"), dtype=torch.float32, device=device)
    return kc, kc.clone(), ks, ks.clone()


def _token_rows(st, vals):
    """Every context token's K/V activation row and slot, after the step's
    append (the appended token's row comes from k_new / v_new)."""
    kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
    oracle.append(vals["k_new"], vals["v_new"], st.slot_mapping, kp, vp)
    B = kp.shape[2]
    slots = []
    for s, L in enumerate(st.context_lens.tolist()):
        row = st.block_tables[s]
        slots += [int(row[t // B]) * B + t % B for t in range(L)]
    sl = torch.tensor(slots, dtype=torch.int64)
    blk, off = sl // B, sl % B
    return kp[blk, :, off].contiguous(), vp[blk, :, off].contiguous(), sl


def build_caches(kind, st, vals):
    """The same quantized cache built by the oracle (CPU) and the library (GPU)."""
    NB, Hk, B, D = vals["k_pool"].shape
    kr, vr, sl = _token_rows(st, vals)
    ref = _empty_pools(NB, Hk, B, D, "cpu")
    oracle.append_quant(kind, kr, vr, sl, *ref)
    gpu = binding.QuantCache(*_empty_pools(NB, Hk, B, D, "cuda"), kind, kr.dtype)
    binding.append_quant(kr.cuda(), vr.cuda(), sl.cuda(), gpu)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    return ref, gpu


def assert_same_cache(ref, gpu):
    kc, vc, ks, vs = ref
    assert torch.equal(gpu.k_codes.cpu(), kc) and torch.equal(gpu.v_codes.cpu(), vc)
    # scales bit for bit, NaN sentinels included
    assert torch.equal(gpu.k_scales.cpu().view(torch.int32), ks.view(torch.int32))
    assert torch.equal(gpu.v_scales.cpu().view(torch.int32), vs.view(torch.int32))


def decode_both(kind, st, vals, ref, gpu, num_ctas=0, seq_ids=None):
    scale = 1.0 / math.sqrt(vals["q"].shape[2])
    out = binding.decode_attention_quant(vals["q"].cuda(), gpu, st.block_tables.cuda(),
                                         st.context_lens.cuda(), scale, out_dtype=torch.float32,
                                         num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    got = out.double().cpu().numpy()
    want = oracle.decode_quant(kind, vals["q"], *ref, st.block_tables, st.context_lens, scale,
                               seq_ids=seq_ids)
    if seq_ids is not None:
        got = got[list(seq_ids)]
    return got, want


def assert_close(got, want, what=""):
    assert np.all(np.isfinite(got)), f"non-finite output {what}"
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert err <= TOL, f"max abs err {err:.3e} > {TOL} {what}"


RAGGED = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 1000]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_append_quant_is_bit_exact(kind, dtype):
    spec = W.WorkloadSpec("q", len(RAGGED), 32, 8, 128, 16, dtype, 1.0)
    st, vals = W.make_workload(spec, seed=51, lengths=RAGGED)
    ref, gpu = build_caches(kind, st, vals)
    assert_same_cache(ref, gpu)


@pytest.mark.parametrize("kind", KINDS)
def test_append_quant_ties_and_zero_rows(kind):
    # rows whose largest element makes the scale exactly 1, holding exact
    # rounding ties, and an all-zero row
    qmax = 127.0 if kind == "int8" else 448.0
    if kind == "int8":
        ties = np.arange(-120.5, 120.5, 1.0)
    else:
        v = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
        m = (v[1:] + v[:-1]) / 2
        ties = np.concatenate([m, -m])
    D = 128
    rows = []
    for i in range(0, len(ties), D - 1):
        r = np.zeros(D)
        chunk = ties[i:i + D - 1]
        r[0] = qmax
        r[1:1 + len(chunk)] = chunk
        rows.append(r)
    rows.append(np.zeros(D))
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.float16)
    assert torch.equal(x.double(), torch.tensor(np.stack(rows)))   # all exact in fp16
    n = x.shape[0]
    kn = x.reshape(n, 1, D)
    vn = -kn
    sl = torch.arange(n, dtype=torch.int64)
    NB = (n + 15) // 16
    ref = _empty_pools(NB, 1, 16, D, "cpu")
    oracle.append_quant(kind, kn, vn, sl, *ref)
    gpu = binding.QuantCache(*_empty_pools(NB, 1, 16, D, "cuda"), kind, torch.float16)
    binding.append_quant(kn.cuda(), vn.cuda(), sl.cuda(), gpu)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    assert_same_cache(ref, gpu)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("dtype,Hq,Hk,B", [("bf16", 32, 8, 16), ("f16", 8, 8, 16),
                                           ("bf16", 64, 8, 8), ("f16", 40, 2, 32),
                                           ("bf16", 16, 8, 16),
                                           # 3, 5 and 6 q heads a kv head: the E4M3
                                           # tensor-core variants' partial units (a
                                           # second PV product; scores on 32 columns)
                                           ("bf16", 24, 8, 16), ("f16", 40, 8, 16),
                                           ("bf16", 48, 8, 16)])
def test_decode_quant_matches_oracle(kind, dtype, Hq, Hk, B):
    spec = W.WorkloadSpec("q", len(RAGGED), Hq, Hk, 128, B, dtype, 1.0)
    st, vals = W.make_workload(spec, seed=52, lengths=RAGGED)
    ref, gpu = build_caches(kind, st, vals)
    got, want = decode_both(kind, st, vals, ref, gpu, num_ctas=9)
    assert_close(got, want, f"{kind} {dtype} {Hq}/{Hk} B{B}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("num_ctas", [0, 1, 3, 64, 600])
def test_decode_quant_ctas(kind, num_ctas):
    spec = W.WorkloadSpec("q", len(RAGGED), 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=53, lengths=RAGGED)
    ref, gpu = build_caches(kind, st, vals)
    got, want = decode_both(kind, st, vals, ref, gpu, num_ctas=num_ctas)
    assert_close(got, want, f"ctas={num_ctas}")


@pytest.mark.parametrize("kind", KINDS)
def test_decode_quant_large_values(kind):
    # activations far outside the fp16 range of q and of p * scale: the kernel
    # scales q heads by powers of two and normalises the V scales per tile
    spec = W.WorkloadSpec("q", 4, 16, 4, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=54, lengths=[70, 300, 1, 129])
    vals = dict(vals)
    big = torch.tensor(1e7, dtype=torch.float32)      # V scales ~2e5: p * s_v > fp16 max
    vals["q"] = (vals["q"].float() * 1e5).to(torch.bfloat16)   # |q| > fp16 max
    vals["k_pool"] = (vals["k_pool"].float() * 1e-4).to(torch.bfloat16)
    vals["k_new"] = (vals["k_new"].float() * 1e-4).to(torch.bfloat16)
    vals["v_pool"] = (vals["v_pool"].float() * big).to(torch.bfloat16)
    vals["v_new"] = (vals["v_new"].float() * big).to(torch.bfloat16)
    ref, gpu = build_caches(kind, st, vals)
    got, want = decode_both(kind, st, vals, ref, gpu, num_ctas=5)
    rel = np.max(np.abs(got - want)) / np.max(np.abs(want))
    assert np.all(np.isfinite(got)) and rel < 1e-4, rel


@pytest.mark.parametrize("kind", KINDS)
def test_decode_quant_llama_workload(kind):
    # every sequence and head of the Llama-shaped workload
    st, vals = W.make_workload(1, seed=0)
    ref, gpu = build_caches(kind, st, vals)
    got, want = decode_both(kind, st, vals, ref, gpu)
    assert_close(got, want, "llama workload")


@pytest.mark.parametrize("kind", KINDS)
def test_decode_quant_long_single_segments(kind):
    # one 131072-token context on 8 CTAs: each CTA runs one segment of about
    # 1000 tiles, so any error that grows with the tiles accumulated in one
    # segment shows (the int8 codes' bias in the PV accumulators); outputs are
    # small here (~0.006), so the bound is tight in relative terms
    spec = W.WorkloadSpec("q", 1, 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=58, lengths=[131072])
    ref, gpu = build_caches(kind, st, vals)
    got, want = decode_both(kind, st, vals, ref, gpu, num_ctas=8)
    assert_close(got, want, "one 131072-token context, 8 CTAs")
    rel = float(np.max(np.abs(got - want)) / np.max(np.abs(want)))
    assert rel < 2e-2, f"max abs err / max |out| = {rel:.2e}"


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("num_ctas", [0, 7])
def test_decode_quant_many_short_sequences(kind, num_ctas):
    # 300 short ragged contexts: many units per CTA, most of them whole
    rng = np.random.default_rng(57)
    lens = rng.integers(1, 200, size=300).tolist()
    lens[255], lens[256] = 129, 1
    spec = W.WorkloadSpec("q", len(lens), 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=57, lengths=lens)
    ref, gpu = build_caches(kind, st, vals)
    got, want = decode_both(kind, st, vals, ref, gpu, num_ctas=num_ctas)
    assert_close(got, want, f"{len(lens)} sequences, ctas={num_ctas}")


@pytest.mark.parametrize("kind", KINDS)
def test_decode_quant_tables_ready_matches_default(kind):
    # quantizing append -> decode steps with the decode reading tables and
    # lengths while the append may still run: the same bits as the default
    spec = W.WorkloadSpec("q", 5, 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=57, lengths=[0, 300, 129, 1000, 1])
    _, gpu = build_caches(kind, st, vals)
    dev = "cuda"
    q, kn, vn = vals["q"].to(dev), vals["k_new"].to(dev), vals["v_new"].to(dev)
    tab, lens, sl = st.block_tables.to(dev), st.context_lens.to(dev), st.slot_mapping.to(dev)
    scale = 1.0 / math.sqrt(128)
    outs = []
    # pending_tail 1: every row but the appended one is gathered while the
    # append may still run
    # inputs_ready: the append reads and quantizes its rows before it waits
    # for the preceding decode, and only its stores wait
    for ready, pend, inp in ((False, 0, False), (True, 0, False), (True, 1, False),
                             (True, 0, True), (True, 1, True)):
        for _ in range(3):
            binding.append_quant(kn, vn, sl, gpu, inputs_ready=inp)
            out = binding.decode_attention_quant(q, gpu, tab, lens, scale, out_dtype=torch.float32,
                                                 num_ctas=7, tables_ready=ready,
                                                 pending_tail=pend)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    assert torch.all(outs[1][0] == 0)


@pytest.mark.parametrize("kind", KINDS)
def test_block_copy_quant_is_byte_exact(kind):
    spec = W.WorkloadSpec("q", 3, 8, 2, 128, 16, "f16", 1.0, pool_ratio=2.0)
    st, vals = W.make_workload(spec, seed=55, lengths=[40, 17, 90])
    ref, gpu = build_caches(kind, st, vals)
    NB = gpu.k_codes.shape[0]
    free = sorted(set(range(NB)) - set(st.block_tables[st.block_tables >= 0].tolist()))
    assert len(free) >= 2
    used = st.block_tables[0, :2].tolist()
    pairs = [[used[0], free[0]], [used[1], free[1]]]
    binding.block_copy_quant(pairs, gpu)
    torch.cuda.synchronize()
    for src, dst in pairs:
        for t in (gpu.k_codes, gpu.v_codes):
            assert torch.equal(t[dst].cpu(), t[src].cpu())
        for t in (gpu.k_scales, gpu.v_scales):
            assert torch.equal(t[dst].cpu().view(torch.int32), t[src].cpu().view(torch.int32))
    with pytest.raises(binding.PkvError):
        binding.block_copy_quant([[used[0], free[0]], [used[1], free[0]]], gpu)


@pytest.mark.parametrize("kind", KINDS)
def test_append_quant_inputs_ready_is_bit_exact(kind):
    # the inputs-ready form (rows quantized before the wait on the preceding
    # kernel, several rows per warp when the grid is full) writes the same
    # codes and scales as the oracle
    # 7695 tokens x 8 kv heads: more rows than the 4096 x 8 warps of a full grid
    lengths = RAGGED + [3000, 2000]
    spec = W.WorkloadSpec("q", len(lengths), 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=58, lengths=lengths)
    NB, Hk, B, D = vals["k_pool"].shape
    kr, vr, sl = _token_rows(st, vals)
    ref = _empty_pools(NB, Hk, B, D, "cpu")
    oracle.append_quant(kind, kr, vr, sl, *ref)
    gpu = binding.QuantCache(*_empty_pools(NB, Hk, B, D, "cuda"), kind, kr.dtype)
    binding.append_quant(kr.cuda(), vr.cuda(), sl.cuda(), gpu, inputs_ready=True)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    assert_same_cache(ref, gpu)


def test_append_quant_out_of_pool_slot_sets_error_word():
    gpu = binding.QuantCache.empty(2, 1, 16, 128, "int8", torch.float16)
    kn = torch.randn(2, 1, 128, device="cuda").to(torch.float16)
    binding.get_error()
    binding.append_quant(kn, kn, torch.tensor([0, 2 * 16], device="cuda"), gpu)
    assert binding.get_error() == binding.DEVERR_SLOT
    binding.append_quant(kn, kn, torch.tensor([0, 2 * 16], device="cuda"), gpu, inputs_ready=True)
    assert binding.get_error() == binding.DEVERR_SLOT


def _base_and_step(kind, dtype, Hq, Hk, B, lengths, seed):
    """A cache holding every context row but each sequence's newest, built the
    same way on both sides, and that step's inputs."""
    spec = W.WorkloadSpec("qf", len(lengths), Hq, Hk, 128, B, dtype, 1.0)
    st, vals = W.make_workload(spec, seed=seed, lengths=lengths)
    NB, Hk_, B_, D = vals["k_pool"].shape
    kr, vr, sl = _token_rows(st, vals)
    keep = ~torch.isin(sl, st.slot_mapping)          # not the newest rows
    ref = _empty_pools(NB, Hk_, B_, D, "cpu")
    oracle.append_quant(kind, kr[keep], vr[keep], sl[keep], *ref)
    gpu = binding.QuantCache(*_empty_pools(NB, Hk_, B_, D, "cuda"), kind, kr.dtype)
    binding.append_quant(kr[keep].cuda(), vr[keep].cuda(), sl[keep].cuda(), gpu)
    torch.cuda.synchronize()
    return st, vals, ref, gpu


def _clone_cache(c):
    return binding.QuantCache(c.k_codes.clone(), c.v_codes.clone(), c.k_scales.clone(),
                              c.v_scales.clone(), c.code, c.act_dtype)


@pytest.mark.parametrize("kind,dtype,Hq,Hk,B", [("fp8_e4m3", "bf16", 32, 8, 16),
                                               ("fp8_e4m3", "f16", 64, 8, 8),
                                               ("fp8_e4m3", "bf16", 16, 8, 32),
                                               ("fp8_e4m3", "f16", 40, 2, 16),
                                               ("int8", "bf16", 32, 8, 16)])
@pytest.mark.parametrize("num_ctas", [0, 5, 300])
def test_append_decode_attention_quant(kind, dtype, Hq, Hk, B, num_ctas):
    # one step: the newest rows quantized into their slots (found from the
    # tables and lengths), then the decode. Pools bit-exact and output bitwise
    # equal to pkv_append_quant + pkv_decode_attention_quant, and within
    # tolerance of the oracle's append and decode
    st, vals, ref, base = _base_and_step(kind, dtype, Hq, Hk, B, RAGGED, seed=61)
    scale = 1.0 / math.sqrt(128)
    q, kn, vn = vals["q"].cuda(), vals["k_new"].cuda(), vals["v_new"].cuda()
    tab, lens = st.block_tables.cuda(), st.context_lens.cuda()
    sep, one = _clone_cache(base), _clone_cache(base)
    binding.append_quant(kn, vn, st.slot_mapping.cuda(), sep)
    want_gpu = binding.decode_attention_quant(q, sep, tab, lens, scale, out_dtype=torch.float32,
                                              num_ctas=num_ctas)
    got = binding.append_decode_attention_quant(q, kn, vn, one, tab, lens, scale,
                                                out_dtype=torch.float32, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    assert torch.equal(one.k_codes.cpu(), sep.k_codes.cpu())
    assert torch.equal(one.v_codes.cpu(), sep.v_codes.cpu())
    assert torch.equal(one.k_scales.cpu().view(torch.int32), sep.k_scales.cpu().view(torch.int32))
    assert torch.equal(one.v_scales.cpu().view(torch.int32), sep.v_scales.cpu().view(torch.int32))
    assert torch.equal(got.cpu(), want_gpu.cpu())
    oracle.append_quant(kind, vals["k_new"], vals["v_new"], st.slot_mapping, *ref)
    assert_same_cache(ref, one)
    want = oracle.decode_quant(kind, vals["q"], *ref, st.block_tables, st.context_lens, scale)
    assert_close(got.double().cpu().numpy(), want, f"{kind} {dtype} {Hq}/{Hk} B{B}")


@pytest.mark.parametrize("kind", KINDS)
def test_append_decode_attention_quant_chain(kind):
    # steps in a row on one cache with the decode reading tables and lengths
    # early and gathering all but the newest rows at once: the same bits each step
    st, vals, ref, base = _base_and_step(kind, "bf16", 32, 8, 16, [0, 300, 129, 1000, 1], seed=62)
    scale = 1.0 / math.sqrt(128)
    q, kn, vn = vals["q"].cuda(), vals["k_new"].cuda(), vals["v_new"].cuda()
    tab, lens = st.block_tables.cuda(), st.context_lens.cuda()
    outs = []
    for ready, pend in ((False, 0), (True, 1), (True, 2)):
        for _ in range(3):
            out = binding.append_decode_attention_quant(q, kn, vn, base, tab, lens, scale,
                                                        out_dtype=torch.float32, num_ctas=7,
                                                        tables_ready=ready, pending_tail=pend)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    assert torch.all(outs[0][0] == 0)
