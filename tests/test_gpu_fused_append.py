"""pkv_append_decode_attention: the append fused into the decode.

One launch per decode step: each sequence's new K/V row goes to position L - 1
of its context (the slot its block table gives) and the attention runs over
the context including it ("KV-Cache Optimization & PagedAttention for
Long-Context Agents", section "Key KV-Cache Optimization Principles", item 1;
"PagedAttention — Math + Memory Model", section "PagedAttention: blocks and
the block table"). Checked against the oracle's append followed by its decode
(pools byte-exact, output within the decode tolerance), and bit for bit
against the library's own two-launch path (pkv_append + pkv_decode_attention).
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


def _oracle_step(st, vals, scale):
    kp, vp = vals["k_pool"].cpu().clone(), vals["v_pool"].cpu().clone()
    if st.cow_pairs.numel():
        oracle.block_copy(st.cow_pairs, kp, vp)
    oracle.append(vals["k_new"].cpu(), vals["v_new"].cpu(), st.slot_mapping, kp, vp)
    ref = oracle.decode(vals["q"].cpu(), kp, vp, st.block_tables, st.context_lens, scale)
    return ref, kp, vp


def _fused(st, vals, **kw):
    dev = "cuda"
    kp, vp = vals["k_pool"].to(dev).clone(), vals["v_pool"].to(dev).clone()
    if st.cow_pairs.numel():
        binding.block_copy(st.cow_pairs, kp, vp)
    scale = 1.0 / math.sqrt(st.spec.head_dim)
    out = binding.append_decode_attention(vals["q"].to(dev), vals["k_new"].to(dev),
                                          vals["v_new"].to(dev), kp, vp,
                                          st.block_tables.to(dev), st.context_lens.to(dev), scale,
                                          out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    return out, kp, vp


RAGGED = [1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 300, 1000]


@pytest.mark.parametrize("num_ctas", [0, 1, 3, 7, 64, 600])
def test_fused_ragged_ctas(num_ctas):
    spec = W.WorkloadSpec("fused", len(RAGGED), 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=31, lengths=RAGGED)
    binding.get_error()
    out, kp, vp = _fused(st, vals, num_ctas=num_ctas)
    assert binding.get_error() == 0
    ref, kp_o, vp_o = _oracle_step(st, vals, 1.0 / math.sqrt(128))
    assert torch.equal(_bits(kp.cpu()), _bits(kp_o)) and torch.equal(_bits(vp.cpu()), _bits(vp_o))
    err = float(np.abs(out.double().cpu().numpy() - ref).max())
    assert err <= 2e-3, err


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("Hq,Hk,D,B", [(4, 4, 64, 16), (8, 2, 64, 8), (16, 1, 128, 32),
                                        (12, 4, 128, 8), (64, 2, 128, 16), (40, 40, 128, 16)])
def test_fused_shapes_and_dtypes(dtype, Hq, Hk, D, B):
    spec = W.WorkloadSpec("fused", 5, Hq, Hk, D, B, dtype, 1.0)
    st, vals = W.make_workload(spec, seed=32, lengths=[1, 5, 70, 129, 450])
    binding.get_error()
    out, kp, vp = _fused(st, vals, num_ctas=5)
    assert binding.get_error() == 0
    ref, kp_o, vp_o = _oracle_step(st, vals, 1.0 / math.sqrt(D))
    assert torch.equal(_bits(kp.cpu()), _bits(kp_o)) and torch.equal(_bits(vp.cpu()), _bits(vp_o))
    err = float(np.abs(out.double().cpu().numpy() - ref).max())
    assert err <= TOL[dtype], err


@pytest.mark.parametrize("consumer", [1, 2])
@pytest.mark.parametrize("opts", [dict(), dict(tables_ready=True),
                                  dict(tables_ready=True, pending_tail=1),
                                  dict(tables_ready=True, pending_tail=5)])
def test_fused_equals_append_then_decode(consumer, opts):
    # the same bits as pkv_append followed by pkv_decode_attention, zero-length
    # sequences included
    spec = W.WorkloadSpec("fused", 7, 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=33, lengths=[0, 700, 65, 0, 1, 2048, 4096])
    dev = "cuda"
    scale = 1.0 / math.sqrt(128)
    kp, vp = vals["k_pool"].to(dev).clone(), vals["v_pool"].to(dev).clone()
    binding.append(vals["k_new"].to(dev), vals["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    sep = binding.decode_attention(vals["q"].to(dev), kp, vp, st.block_tables.to(dev),
                                   st.context_lens.to(dev), scale, out_dtype=torch.float32,
                                   num_ctas=9, consumer=consumer)
    out, kp2, vp2 = _fused(st, vals, num_ctas=9, consumer=consumer, **opts)
    assert binding.get_error() == 0
    assert torch.equal(out, sep)
    assert torch.equal(_bits(kp), _bits(kp2)) and torch.equal(_bits(vp), _bits(vp2))
    assert torch.all(out[0] == 0) and torch.all(out[3] == 0)


def test_fused_copy_on_write_workload_small():
    spec = W.WorkloadSpec("fused_cow", 5, 32, 8, 128, 16, "f16", 1.0, shared_prefix=256,
                          suffix_lo=0, suffix_hi=300, cow=True)
    st, vals = W.make_workload(spec, seed=34)
    assert st.cow_pairs.shape[0] == 4
    out, kp, vp = _fused(st, vals, num_ctas=11, tables_ready=True)
    assert binding.get_error() == 0
    ref, kp_o, vp_o = _oracle_step(st, vals, 1.0 / math.sqrt(128))
    assert torch.equal(_bits(kp.cpu()), _bits(kp_o)) and torch.equal(_bits(vp.cpu()), _bits(vp_o))
    assert float(np.abs(out.double().cpu().numpy() - ref).max()) <= 2e-3


def test_fused_serving_loop_on_one_cache():
    # three steps on one cache: each step's context is one token longer and
    # its newest row is the call's own; the row the previous call appended is
    # read from the pool, so pending_tail 2 (that row may still be in flight)
    g = torch.Generator().manual_seed(35)
    final = [3, 16, 17, 64, 129, 1000, 2050]
    spec = W.WorkloadSpec("loop", len(final), 32, 8, 128, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=35, lengths=final)
    dev = "cuda"
    scale = 1.0 / math.sqrt(128)
    kp, vp = vals["k_pool"].to(dev).clone(), vals["v_pool"].to(dev).clone()
    kp_o, vp_o = vals["k_pool"].clone(), vals["v_pool"].clone()
    q, tab = vals["q"].to(dev), st.block_tables.to(dev)
    ws = binding.alloc_workspace(kp, 32)
    binding.get_error()
    for back in (2, 1, 0):
        lens = (st.context_lens - back).to(torch.int32)
        kn = (torch.randn(vals["k_new"].shape, generator=g)).to(torch.bfloat16)
        vn = (torch.randn(vals["v_new"].shape, generator=g)).to(torch.bfloat16)
        out = binding.append_decode_attention(q, kn.to(dev), vn.to(dev), kp, vp, tab,
                                              lens.to(dev), scale, out_dtype=torch.float32,
                                              workspace=ws, tables_ready=True, pending_tail=2)
        pos = lens.long() - 1
        slots = tab.cpu().long()[torch.arange(len(final)), pos // 16] * 16 + pos % 16
        oracle.append(kn, vn, slots, kp_o, vp_o)
        ref = oracle.decode(vals["q"], kp_o, vp_o, st.block_tables, lens, scale)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        err = float(np.abs(out.double().cpu().numpy() - ref).max())
        assert err <= 2e-3, (back, err)
    assert torch.equal(_bits(kp.cpu()), _bits(kp_o)) and torch.equal(_bits(vp.cpu()), _bits(vp_o))


def test_fused_bad_block_id_sets_error_word():
    spec = W.WorkloadSpec("fused", 2, 8, 2, 64, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=36, lengths=[40, 20])
    bt = st.block_tables.clone()
    bt[0, 2] = st.num_blocks + 5          # the block holding token 39, the new one
    dev = "cuda"
    kp, vp = vals["k_pool"].to(dev).clone(), vals["v_pool"].to(dev).clone()
    before = kp.clone()
    binding.get_error()
    out = binding.append_decode_attention(vals["q"].to(dev), vals["k_new"].to(dev),
                                          vals["v_new"].to(dev), kp, vp, bt.to(dev),
                                          st.context_lens.to(dev), 0.125, out_dtype=torch.float32)
    assert binding.get_error() & binding.DEVERR_BLOCK_ID
    assert torch.isfinite(out).all()
    # sequence 1 appended its row; sequence 0's row went nowhere
    changed = (_bits(kp) != _bits(before)).any(dim=-1).nonzero().tolist()
    s1 = int(st.slot_mapping[1])
    assert sorted(changed) == sorted([[s1 // 16, h, s1 % 16] for h in range(2)])


def test_fused_arguments_are_checked():
    spec = W.WorkloadSpec("fused", 2, 8, 2, 64, 16, "bf16", 1.0)
    st, vals = W.make_workload(spec, seed=37, lengths=[10, 20])
    dev = "cuda"
    args = [vals["q"].to(dev), vals["k_new"].to(dev), vals["v_new"].to(dev),
            vals["k_pool"].to(dev), vals["v_pool"].to(dev), st.block_tables.to(dev),
            st.context_lens.to(dev), 0.1]
    with pytest.raises(binding.PkvError):
        binding.append_decode_attention(*args, pending_tail=1)        # without tables_ready
    kn_bad = torch.empty(2 * 2 * 64 + 1, dtype=torch.bfloat16, device=dev)[1:].view(2, 2, 64)
    with pytest.raises(binding.PkvError):
        binding.append_decode_attention(args[0], kn_bad, *args[2:])   # misaligned k_new
