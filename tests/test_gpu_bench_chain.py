"""The benchmark's own chain of calls, checked against the oracle.

bench.py times the Llama-3-8B-shaped decode step (64 sequences, 32 q / 8 kv
heads, head_dim 128, bf16, block size 16, context lengths U[512, 4096]) as a
chain of prepared C-ABI calls over three resident cache copies used in turn,
with the launch-overlap promises it makes there (the append reading its
inputs before its wait, the decode reading tables and lengths early and
gathering every row but the appended one early). This test builds that chain
with bench.py's own classes, runs it for several steps, and compares every
output element of every cache copy, and every byte of each copy's pools, with
the oracle: paging and launch overlap move bytes, not results ("PagedAttention
— Math + Memory Model", sections "The operating-system analogy" and
"PagedAttention: blocks and the block table"). The same holds for the
8-bit steps bench.py times with --kv-quant (the quantizing append reading and
quantizing its rows before its wait, the decode reading tables and lengths
early): codes and scales bit for bit, outputs within tolerance of the
oracle's own quantized cache.
"""
import math

import pytest
import torch

import bench
from oracle import oracle
from paged_kv_cache_47_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()
    yield


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("steps", [7])
def test_bench_chain_matches_oracle(steps):
    dev = torch.device("cuda")
    spec = W.SPECS[bench.WORKLOAD_INDEX]
    st = W.make_structure(spec, 0)
    vals = W.make_values(st, 0, device=dev)
    host = {k: v.cpu() for k, v in vals.items()}
    scale = 1.0 / math.sqrt(spec.head_dim)
    tables, lens = st.block_tables.to(dev), st.context_lens.to(dev)
    slots = st.slot_mapping.to(dev)
    S, Hq, D = vals["q"].shape
    base = bench.Pools16(vals["k_pool"], vals["v_pool"])
    copies = [base] + [base.clone() for _ in range(2)]
    outs = [torch.full((S, Hq, D), float("nan"), dtype=vals["q"].dtype, device=dev)
            for _ in copies]
    wss = [c.workspace(Hq) for c in copies]
    calls = [c.prepared(vals["q"], vals["k_new"], vals["v_new"], slots, tables, lens, scale, o,
                        w, pending_tail=1)
             for c, o, w in zip(copies, outs, wss)]
    stream = torch.cuda.current_stream()
    binding.get_error()
    for i in range(steps):
        app, dec = calls[i % len(calls)]
        if app is not None:          # a separate append (the fused step has none)
            app(stream)
        dec(stream)
    torch.cuda.synchronize()
    assert binding.get_error() == 0

    oracle.append(host["k_new"], host["v_new"], st.slot_mapping, host["k_pool"], host["v_pool"])
    ref = oracle.decode(host["q"], host["k_pool"], host["v_pool"], st.block_tables,
                        st.context_lens, scale)
    kp_ref, vp_ref = host["k_pool"].to(dev), host["v_pool"].to(dev)
    for c, o in zip(copies, outs):
        assert torch.equal(_bits(c.kp), _bits(kp_ref)) and torch.equal(_bits(c.vp), _bits(vp_ref))
        got = o.double().cpu().numpy()
        err = float(abs(got - ref).max())
        assert err <= 2e-3, f"max abs err {err:.3e}"


@pytest.mark.parametrize("kind", ["fp8_e4m3", "int8"])
def test_bench_chain_8bit_matches_oracle(kind, steps=7):
    dev = torch.device("cuda")
    spec = W.SPECS[bench.WORKLOAD_INDEX]
    st = W.make_structure(spec, 0)
    vals = W.make_values(st, 0, device=dev)
    scale = 1.0 / math.sqrt(spec.head_dim)
    tables, lens = st.block_tables.to(dev), st.context_lens.to(dev)
    slots = st.slot_mapping.to(dev)
    S, Hq, D = vals["q"].shape
    base = bench.PoolsQ.fill(kind, st, vals, dev)
    copies = [base] + [base.clone() for _ in range(2)]
    outs = [torch.full((S, Hq, D), float("nan"), dtype=vals["q"].dtype, device=dev)
            for _ in copies]
    wss = [c.workspace(Hq) for c in copies]
    calls = [c.prepared(vals["q"], vals["k_new"], vals["v_new"], slots, tables, lens, scale, o,
                        w)
             for c, o, w in zip(copies, outs, wss)]
    stream = torch.cuda.current_stream()
    binding.get_error()
    for i in range(steps):
        app, dec = calls[i % len(calls)]
        app(stream)
        dec(stream)
    torch.cuda.synchronize()
    assert binding.get_error() == 0

    # the oracle quantizes every context row (the appended ones included) itself
    h = bench.host_inputs_from_generator(st, 0, dev, kind)
    ref = oracle.decode_quant(kind, h["q"], h["k_codes"], h["v_codes"], h["k_scales"],
                              h["v_scales"], st.block_tables, st.context_lens, scale)
    for c, o in zip(copies, outs):
        cache = c.cache
        assert torch.equal(cache.k_codes.cpu(), h["k_codes"])
        assert torch.equal(cache.v_codes.cpu(), h["v_codes"])
        assert torch.equal(cache.k_scales.cpu().view(torch.int32), h["k_scales"].view(torch.int32))
        assert torch.equal(cache.v_scales.cpu().view(torch.int32), h["v_scales"].view(torch.int32))
        got = o.double().cpu().numpy()
        err = float(abs(got - ref).max())
        assert err <= 2e-3, f"{kind}: max abs err {err:.3e}"


def test_bench_chain_flat_matches_oracle(steps=7):
    # bench.py --flat: three flat caches (one virtual span per sequence), the
    # flat append then the flat decode, with the decode reading lengths early
    # and gathering every row but the appended one early
    dev = torch.device("cuda")
    spec = W.SPECS[bench.WORKLOAD_INDEX]
    st = W.make_structure(spec, 0)
    vals = W.make_values(st, 0, device=dev)
    host = {k: v.cpu() for k, v in vals.items()}
    scale = 1.0 / math.sqrt(spec.head_dim)
    tables, lens = st.block_tables.to(dev), st.context_lens.to(dev)
    slots = st.slot_mapping.to(dev)
    S, Hq, D = vals["q"].shape
    copies = [bench.PoolsFlat.fill(st, vals, dev) for _ in range(3)]
    outs = [torch.full((S, Hq, D), float("nan"), dtype=vals["q"].dtype, device=dev)
            for _ in copies]
    wss = [c.workspace(Hq) for c in copies]
    calls = [c.prepared(vals["q"], vals["k_new"], vals["v_new"], slots, tables, lens, scale, o,
                        w, pending_tail=1)
             for c, o, w in zip(copies, outs, wss)]
    stream = torch.cuda.current_stream()
    binding.get_error()
    for i in range(steps):
        app, dec = calls[i % len(calls)]
        app(stream)
        dec(stream)
    torch.cuda.synchronize()
    assert binding.get_error() == 0

    oracle.append(host["k_new"], host["v_new"], st.slot_mapping, host["k_pool"], host["v_pool"])
    ref = oracle.decode(host["q"], host["k_pool"], host["v_pool"], st.block_tables,
                        st.context_lens, scale)
    for o in outs:
        got = o.double().cpu().numpy()
        err = float(abs(got - ref).max())
        assert err <= 2e-3, f"flat: max abs err {err:.3e}"
