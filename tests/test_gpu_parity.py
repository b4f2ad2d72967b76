"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Append and block copy must be byte-exact. Decode attention must match the fp64
oracle within max-abs 2e-3 for fp16/bf16 K/V and 1e-5 for fp32 K/V (the
tolerance of the decode-attention target). Every test compares every output
element: small cases cover the edge cases, and the five workloads run at full
size (the long-context one at block sizes 8, 16 and 32). The chain of calls
the benchmark times (rotating cache copies and the launch-overlap options) is
checked against the oracle in test_gpu_bench_chain.py.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_cache_47_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()
    yield


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def run_step(st, vals, *, out_dtype=None, num_ctas=0, consumer=0, check_pools=True):
    """Copy-on-write + append + decode on the GPU and in the oracle; returns
    (gpu_out as float64 numpy, oracle_out, GPU pools)."""
    dev = "cuda"
    spec = st.spec
    scale = 1.0 / math.sqrt(spec.head_dim)
    # oracle side (CPU copies of the inputs)
    kp_o = vals["k_pool"].detach().cpu().clone()
    vp_o = vals["v_pool"].detach().cpu().clone()
    if st.cow_pairs.numel():
        oracle.block_copy(st.cow_pairs, kp_o, vp_o)
    oracle.append(vals["k_new"].cpu(), vals["v_new"].cpu(), st.slot_mapping, kp_o, vp_o)
    ref = oracle.decode(vals["q"].cpu(), kp_o, vp_o, st.block_tables, st.context_lens, scale)
    # CUDA side
    kp = vals["k_pool"].to(dev).clone()
    vp = vals["v_pool"].to(dev).clone()
    if st.cow_pairs.numel():
        binding.block_copy(st.cow_pairs, kp, vp)
    binding.append(vals["k_new"].to(dev), vals["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    out = binding.decode_attention(vals["q"].to(dev), kp, vp, st.block_tables.to(dev),
                                   st.context_lens.to(dev), scale, out_dtype=out_dtype,
                                   num_ctas=num_ctas, consumer=consumer)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    if check_pools:
        assert torch.equal(_bits(kp.cpu()), _bits(kp_o)), "K pool differs after append/copy"
        assert torch.equal(_bits(vp.cpu()), _bits(vp_o)), "V pool differs after append/copy"
    return out.double().cpu().numpy(), ref, (kp, vp)


def assert_close(got, ref, dtype, what=""):
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"non-finite output {what}"
    m = float(err.max()) if err.size else 0.0
    assert m <= TOL[dtype], f"max abs err {m:.3e} > {TOL[dtype]} {what}"
    return m


def spec_like(i, **kw):
    return W.SPECS[i].__class__(**{**W.SPECS[i].__dict__, **kw})


# ----------------------------------------------------------------- small cases
RAGGED = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 300, 1000]


def test_tiny_workload_full():
    st, vals = W.make_workload(0, seed=0)
    got, ref, _ = run_step(st, vals)
    assert_close(got, ref, "f32")


@pytest.mark.parametrize("num_ctas", [0, 1, 3, 7, 64, 600])
def test_gqa4_bf16_ragged_ctas(num_ctas):
    spec = spec_like(1, num_seqs=len(RAGGED))
    st, vals = W.make_workload(spec, seed=1, lengths=RAGGED)
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32, num_ctas=num_ctas)
    assert_close(got, ref, "bf16", f"ctas={num_ctas}")


def test_workspace_reuse_keeps_counters_zero():
    """One zero-filled workspace, sized for the largest launch, serves calls
    with different batches, head groupings and CTA counts in a row (a call
    with more CTAs than the one before it finds that call's partials just past
    the counters it used). Each call must match the oracle, which needs the
    counters to read zero when it starts, and must leave every arrival counter
    of the buffer at zero."""
    cases = [(41, 32, 8, 152, [1, 70, 513, 1500, 4096, 64, 2000, 333]),
             (42, 32, 8, 7, [3000, 17, 900]),
             (43, 16, 16, 600, [65, 129, 5, 64]),
             (44, 64, 8, 300, [2048, 1, 777, 4000, 4000]),
             (41, 32, 8, 152, [1, 70, 513, 1500, 4096, 64, 2000, 333])]
    max_c = max(c[3] for c in cases)
    ws = None
    for seed, hq, hk, C, lengths in cases:
        spec = W.WorkloadSpec("reuse", len(lengths), hq, hk, 128, 16, "bf16", 1.0)
        st, vals = W.make_workload(spec, seed=seed, lengths=lengths)
        dev = "cuda"
        kp, vp = vals["k_pool"].to(dev), vals["v_pool"].to(dev)
        if ws is None:   # heads-per-unit is 16 at most: size for the largest layout
            ws = binding.alloc_workspace(kp, 16 * hk, max_c)
        binding.append(vals["k_new"].to(dev), vals["v_new"].to(dev), st.slot_mapping.to(dev),
                       kp, vp)
        scale = 1.0 / math.sqrt(128)
        out = binding.decode_attention(vals["q"].to(dev), kp, vp, st.block_tables.to(dev),
                                       st.context_lens.to(dev), scale, out_dtype=torch.float32,
                                       workspace=ws, num_ctas=C)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        kp_o, vp_o = vals["k_pool"].clone(), vals["v_pool"].clone()
        oracle.append(vals["k_new"], vals["v_new"], st.slot_mapping, kp_o, vp_o)
        ref = oracle.decode(vals["q"], kp_o, vp_o, st.block_tables, st.context_lens, scale)
        assert_close(out.double().cpu().numpy(), ref, "bf16", f"ctas={C}")
        counters = ws[: 4096 * 16].view(torch.int32)   # [4096 CTAs][4 math warps]
        assert int(counters.abs().sum()) == 0, "arrival counters left non-zero"


@pytest.mark.parametrize("consumer", [1, 2])
@pytest.mark.parametrize("dtype,Hq,Hk,D", [("bf16", 32, 8, 128), ("f16", 8, 8, 128),
                                            ("f16", 16, 8, 128), ("bf16", 24, 8, 128),
                                            ("bf16", 64, 8, 128), ("f16", 40, 2, 128),
                                            ("f16", 4, 4, 64), ("bf16", 8, 4, 64)])
def test_forced_consumers(consumer, dtype, Hq, Hk, D):
    spec = W.WorkloadSpec("t", 5, Hq, Hk, D, 16, dtype, 1.0)
    st, vals = W.make_workload(spec, seed=2, lengths=[1, 40, 64, 333, 777])
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32, consumer=consumer, num_ctas=9)
    assert_close(got, ref, dtype, f"consumer={consumer}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("Hq,Hk,D,B", [(4, 4, 64, 16), (8, 2, 64, 8), (16, 1, 128, 32),
                                        (12, 4, 128, 8), (20, 1, 64, 16)])
def test_shapes_and_dtypes(dtype, Hq, Hk, D, B):
    spec = W.WorkloadSpec("t", 4, Hq, Hk, D, B, dtype, 1.0)
    st, vals = W.make_workload(spec, seed=3, lengths=[5, 70, 129, 450])
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32, num_ctas=5)
    assert_close(got, ref, dtype)


def test_mha_fp16_small():
    spec = spec_like(2, num_seqs=6)
    st, vals = W.make_workload(spec, seed=4, lengths=[128, 129, 700, 2048, 1, 64])
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32)
    assert_close(got, ref, "f16")


def test_prefix_sharing_with_copy_on_write_small():
    spec = spec_like(3, num_seqs=5, shared_prefix=256, suffix_lo=0, suffix_hi=300)
    st, vals = W.make_workload(spec, seed=5)
    assert st.cow_pairs.shape[0] == 4
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32, num_ctas=11)
    assert_close(got, ref, "f16")


@pytest.mark.parametrize("B", [8, 16, 32])
def test_long_context_gqa8_small(B):
    spec = spec_like(4, num_seqs=2)
    st, vals = W.make_workload(spec, seed=6, block_size=B, lengths=[3001, 5000])
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32)
    assert_close(got, ref, "bf16", f"B={B}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_long_single_segments(dtype):
    # one 131072-token context on 8 CTAs: each CTA runs one segment of about
    # 2000 tiles, so an error that grew with the tiles accumulated in one
    # segment would show; outputs are small (~0.01), so the relative bound is
    # the tight one
    spec = spec_like(1, num_seqs=1, dtype=dtype)
    st, vals = W.make_workload(spec, seed=9, lengths=[131072])
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32, num_ctas=8, check_pools=False)
    assert_close(got, ref, dtype, "one 131072-token context, 8 CTAs")
    rel = float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))
    assert rel < 2e-2, f"max abs err / max |out| = {rel:.2e}"


def test_zero_length_sequences_give_zeros():
    spec = W.WorkloadSpec("t", 4, 8, 2, 64, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=7, lengths=[0, 33, 0, 90])
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32, num_ctas=4)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert_close(got, ref, "bf16")


@pytest.mark.parametrize("num_ctas", [0, 5])
def test_tables_ready_matches_default(num_ctas):
    # append -> decode steps, the decode reading tables and lengths while the
    # append may still run (programmatic dependent launch): same bits as the
    # default, zero-length sequences included, and equal to the oracle
    spec = W.WorkloadSpec("t", 6, 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=9, lengths=[0, 700, 65, 0, 1, 2048])
    dev = "cuda"
    scale = 1.0 / math.sqrt(128)
    q, kn, vn = vals["q"].to(dev), vals["k_new"].to(dev), vals["v_new"].to(dev)
    tab, lens, sl = st.block_tables.to(dev), st.context_lens.to(dev), st.slot_mapping.to(dev)
    outs = []
    # pending_tail n: the rows below each sequence's last n are gathered while
    # the append may still run; the appended row (the last) waits for it
    for ready, pend in ((False, 0), (True, 0), (True, 1), (True, 3), (True, 64), (False, 0)):
        kp, vp = vals["k_pool"].to(dev).clone(), vals["v_pool"].to(dev).clone()
        ws = binding.alloc_workspace(kp, 32, num_ctas)
        for _ in range(3):
            binding.append(kn, vn, sl, kp, vp)
            out = binding.decode_attention(q, kp, vp, tab, lens, scale, out_dtype=torch.float32,
                                           workspace=ws, num_ctas=num_ctas, tables_ready=ready,
                                           pending_tail=pend)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    _, ref, _ = run_step(st, vals, out_dtype=torch.float32, num_ctas=num_ctas)
    assert_close(outs[1].double().numpy(), ref, "bf16")
    assert torch.all(outs[1][0] == 0) and torch.all(outs[1][3] == 0)


def test_pending_tail_sees_the_appended_row():
    # The appended row dominates the output (large new K along q, distinct V),
    # so a decode that gathered it before the append landed would be far off.
    # Each step appends into a fresh cache copy right before the decode.
    spec = W.WorkloadSpec("t", 8, 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=4, lengths=[1, 17, 64, 65, 300, 1000, 2049, 4096])
    dev = "cuda"
    scale = 1.0 / math.sqrt(128)
    q = vals["q"].to(dev)
    kn = (vals["q"].view(8, 8, 4, 128)[:, :, 0, :] * 4.0).to(torch.bfloat16).to(dev)
    vn = torch.full_like(vals["v_new"], 3.0).to(dev)
    tab, lens, sl = st.block_tables.to(dev), st.context_lens.to(dev), st.slot_mapping.to(dev)
    vals2 = dict(vals, k_new=kn.cpu(), v_new=vn.cpu())
    _, ref, _ = run_step(st, vals2, out_dtype=torch.float32)
    for num_ctas in (0, 3):
        ws = binding.alloc_workspace(vals["k_pool"].to(dev), 32, num_ctas)
        for _ in range(4):
            kp, vp = vals["k_pool"].to(dev), vals["v_pool"].to(dev)
            binding.append(kn, vn, sl, kp, vp)
            out = binding.decode_attention(q, kp, vp, tab, lens, scale, out_dtype=torch.float32,
                                           workspace=ws, num_ctas=num_ctas, tables_ready=True,
                                           pending_tail=1)
            torch.cuda.synchronize()
            assert binding.get_error() == 0
            assert_close(out.cpu().double().numpy(), ref, "bf16")


def test_append_inputs_ready_matches_default():
    # the append reading its inputs before the wait on the preceding kernel
    # (here a decode) writes the same bytes, after that kernel's reads
    spec = W.WorkloadSpec("t", 6, 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=12, lengths=[5, 700, 64, 1, 2049, 300])
    dev = "cuda"
    scale = 1.0 / math.sqrt(128)
    q, kn, vn = vals["q"].to(dev), vals["k_new"].to(dev), vals["v_new"].to(dev)
    tab, lens, sl = st.block_tables.to(dev), st.context_lens.to(dev), st.slot_mapping.to(dev)
    res = []
    for ready in (False, True):
        kp, vp = vals["k_pool"].to(dev), vals["v_pool"].to(dev)
        for _ in range(3):
            binding.append(kn, vn, sl, kp, vp, inputs_ready=ready)
            out = binding.decode_attention(q, kp, vp, tab, lens, scale, out_dtype=torch.float32,
                                           tables_ready=True, pending_tail=int(ready))
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        res.append((kp.cpu(), vp.cpu(), out.cpu()))
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
    _, ref, _ = run_step(st, vals, out_dtype=torch.float32)
    assert_close(res[1][2].double().numpy(), ref, "bf16")


def test_pending_tail_is_checked():
    spec = spec_like(1, num_seqs=2)
    st, vals = W.make_workload(spec, seed=1)
    dev = "cuda"
    args = (vals["q"].to(dev), vals["k_pool"].to(dev), vals["v_pool"].to(dev),
            st.block_tables.to(dev), st.context_lens.to(dev), 0.1)
    with pytest.raises(binding.PkvError):
        binding.decode_attention(*args, pending_tail=1)             # without tables_ready
    with pytest.raises(binding.PkvError):
        binding.decode_attention(*args, tables_ready=True, pending_tail=-1)


def test_native_output_is_rne_of_fp32_output():
    spec = spec_like(1, num_seqs=4)
    st, vals = W.make_workload(spec, seed=8, lengths=[3, 100, 1500, 4096])
    f32, _, _ = run_step(st, vals, out_dtype=torch.float32, check_pools=False)
    b16, ref, _ = run_step(st, vals, out_dtype=torch.bfloat16, check_pools=False)
    rne = torch.from_numpy(f32).float().to(torch.bfloat16).double().numpy()
    assert np.array_equal(b16, rne)


def test_repeated_calls_are_deterministic():
    spec = spec_like(1, num_seqs=5)
    st, vals = W.make_workload(spec, seed=9, lengths=[17, 500, 1200, 64, 4000])
    a, _, _ = run_step(st, vals, out_dtype=torch.float32, check_pools=False)
    b, _, _ = run_step(st, vals, out_dtype=torch.float32, check_pools=False)
    assert np.array_equal(a, b)


def test_many_sequences_chunked_launch():
    # more sequences than one launch carries: the library splits the batch
    spec = W.WorkloadSpec("t", 1100, 8, 8, 64, 16, "f16", 1.0, 1, 40)
    st, vals = W.make_workload(spec, seed=10)
    got, ref, _ = run_step(st, vals, out_dtype=torch.float32)
    assert_close(got, ref, "f16")


# ----------------------------------------------------------------- device-side checks
def test_out_of_range_block_id_sets_error_word():
    spec = W.WorkloadSpec("t", 2, 8, 2, 64, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=11, lengths=[40, 20])
    bt = st.block_tables.clone()
    bt[0, 1] = st.num_blocks + 5
    dev = "cuda"
    kp, vp = vals["k_pool"].to(dev), vals["v_pool"].to(dev)
    binding.append(vals["k_new"].to(dev), vals["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    binding.get_error()
    out = binding.decode_attention(vals["q"].to(dev), kp, vp, bt.to(dev),
                                   st.context_lens.to(dev), 0.125, out_dtype=torch.float32)
    w = binding.get_error()
    assert w & binding.DEVERR_BLOCK_ID
    assert torch.isfinite(out[1]).all()


def test_context_len_past_table_sets_error_word():
    spec = W.WorkloadSpec("t", 2, 8, 2, 64, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=12, lengths=[40, 20])
    cl = st.context_lens.clone()
    cl[1] = 10_000
    dev = "cuda"
    binding.get_error()
    binding.decode_attention(vals["q"].to(dev), vals["k_pool"].to(dev), vals["v_pool"].to(dev),
                             st.block_tables.to(dev), cl.to(dev), 0.125)
    assert binding.get_error() & binding.DEVERR_CONTEXT


def test_append_slot_past_pool_sets_error_word():
    kp = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device="cuda")
    vp = torch.zeros_like(kp)
    kn = torch.ones(2, 2, 64, dtype=torch.float16, device="cuda")
    binding.get_error()
    binding.append(kn, kn, torch.tensor([3, 4 * 16], dtype=torch.int64, device="cuda"), kp, vp)
    assert binding.get_error() & binding.DEVERR_SLOT
    assert torch.all(kp[0, :, 3] == 1) and int((kp != 0).sum()) == 2 * 64


def test_block_copy_leaves_other_blocks_untouched():
    g = torch.Generator().manual_seed(13)
    kp = torch.randn(20, 3, 8, 64, generator=g).to(torch.bfloat16)
    vp = torch.randn(20, 3, 8, 64, generator=g).to(torch.bfloat16)
    pairs = [[1, 5], [7, 2], [19, 0]]
    ko, vo = kp.clone(), vp.clone()
    oracle.block_copy(pairs, ko, vo)
    kg, vg = kp.cuda(), vp.cuda()
    binding.block_copy(pairs, kg, vg)
    assert torch.equal(_bits(kg.cpu()), _bits(ko)) and torch.equal(_bits(vg.cpu()), _bits(vo))


def test_many_block_copy_pairs():
    NB = 600
    kp = torch.arange(NB * 2 * 16 * 64, dtype=torch.float32).view(NB, 2, 16, 64)
    vp = -kp
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(1)).tolist()
    pairs = [[perm[i], perm[i + 300]] for i in range(300)]
    ko, vo = kp.clone(), vp.clone()
    oracle.block_copy(pairs, ko, vo)
    kg, vg = kp.cuda(), vp.cuda()
    binding.block_copy(pairs, kg, vg)
    assert torch.equal(kg.cpu(), ko) and torch.equal(vg.cpu(), vo)


# ----------------------------------------------------------------- full-size workloads
def _full(i, block_size=None, seed=0):
    """Copy-on-write + append + decode of a whole workload at its full size,
    every output element (all sequences, all heads) against the oracle."""
    spec = W.SPECS[i] if block_size is None else W.SPECS[i].with_block_size(block_size)
    st = W.make_structure(spec, seed)
    vals = W.make_values(st, seed, device="cuda")
    dev = "cuda"
    scale = 1.0 / math.sqrt(spec.head_dim)
    kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
    if st.cow_pairs.numel():
        binding.block_copy(st.cow_pairs, kp, vp)
    binding.append(vals["k_new"], vals["v_new"], st.slot_mapping.to(dev), kp, vp)
    out = binding.decode_attention(vals["q"], kp, vp, st.block_tables.to(dev),
                                   st.context_lens.to(dev), scale)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    # oracle on host copies
    kp_o, vp_o = vals["k_pool"].cpu(), vals["v_pool"].cpu()
    if st.cow_pairs.numel():
        oracle.block_copy(st.cow_pairs, kp_o, vp_o)
    oracle.append(vals["k_new"].cpu(), vals["v_new"].cpu(), st.slot_mapping, kp_o, vp_o)
    assert torch.equal(_bits(kp.cpu()), _bits(kp_o)) and torch.equal(_bits(vp.cpu()), _bits(vp_o))
    ref = oracle.decode(vals["q"].cpu(), kp_o, vp_o, st.block_tables, st.context_lens, scale)
    got = out.double().cpu().numpy()
    assert got.shape == ref.shape == (spec.num_seqs, spec.num_q_heads, spec.head_dim)
    return assert_close(got, ref, spec.dtype, f"workload {i} B={spec.block_size}")


@pytest.mark.parametrize("i", [0, 1, 2, 3])
def test_full_workload_every_output(i):
    _full(i)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_full_long_context_every_output(B):
    _full(4, block_size=B)
