"""Prefix-aware decode (pkv_decode_attention_prefix) and the decode's lse_out
option, against the oracle.

The prefix-aware call decodes each group's shared prefix once per unit of
several sharers' heads and each sequence's private suffix on its own, in one
launch, and merges the two by log-sum-exp inside the kernel. It must give the
plain decode's result (the oracle's dense attention over each whole context,
"PagedAttention — Math + Memory Model", section "PagedAttention: blocks and
the block table") within 2e-3, for every output element: groups of sequences
that share leading blocks, sequences in no group, members whose private
suffix is empty, groups larger than one unit, every head grouping and head
size, and shapes outside the one-launch variants (which the library serves
with the plain decode). lse_out must be log2 of each head's softmax
denominator.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_cache_47_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


def _shared_case(lens, groups, dtype="bf16", Hq=32, Hk=8, D=128, B=16, seed=91):
    """Tables drawn by the generator, then each group's members point their
    first `pb` entries at the group's first member's blocks. groups: list of
    (member list, pb)."""
    spec = W.WorkloadSpec("pfx", len(lens), Hq, Hk, D, B, dtype, 1.0, pool_ratio=1.0)
    st, vals = W.make_workload(spec, seed=seed, lengths=lens)
    bt = st.block_tables.clone()
    gos = [-1] * len(lens)
    gpb = []
    for gi, (mem, pb) in enumerate(groups):
        for s in mem:
            bt[s, :pb] = bt[mem[0], :pb]
            gos[s] = gi
        gpb.append(pb)
    kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
    oracle.append(vals["k_new"], vals["v_new"], st.slot_mapping, kp, vp)
    return vals["q"], kp, vp, bt, torch.tensor(lens, dtype=torch.int32), gos, gpb


def _check(q, kp, vp, bt, cl, gos, gpb, tol=2e-3, **kw):
    scale = 1.0 / math.sqrt(q.shape[2])
    want = oracle.decode(q, kp, vp, bt, cl, scale)
    out = binding.decode_attention_prefix(q.cuda(), kp.cuda(), vp.cuda(), bt.cuda(), cl.cuda(),
                                          scale, gos, gpb, out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert binding.get_error() == 0
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - want)))
    assert err <= tol, err
    return out


def _two_groups(B=16):
    # sequences 0-3 share a 5-block prefix (2 ends exactly with it), 4-5 a
    # 3-block prefix, 6 is on its own
    lens = [5 * B + 30, 5 * B + 200, 5 * B, 5 * B + 1, 3 * B + 77, 3 * B + 5, 400]
    return lens, [([0, 1, 2, 3], 5), ([4, 5], 3)]


@pytest.mark.parametrize("num_ctas", [0, 1, 3, 7, 64, 600])
def test_prefix_aware_equals_plain_decode(num_ctas):
    lens, groups = _two_groups()
    _check(*_shared_case(lens, groups), num_ctas=num_ctas)


@pytest.mark.parametrize("dtype,Hq,Hk,D,B", [("bf16", 32, 8, 128, 16), ("f16", 8, 8, 128, 8),
                                              ("bf16", 64, 8, 128, 32), ("f16", 64, 4, 128, 16),
                                              ("bf16", 16, 8, 64, 16), ("f16", 24, 8, 64, 8),
                                              ("bf16", 24, 8, 128, 16)])
def test_prefix_aware_head_groupings(dtype, Hq, Hk, D, B):
    # MHA (8 members a unit), GQA 3 / 4 / 8 / 16, head size 64 with 2 heads per
    # kv head (one launch) and 3 (the plain decode serves it); a 10-member
    # group spans several prefix units
    lens = [6 * B + k * 37 for k in range(10)] + [6 * B, 2 * B + 3, 900]
    groups = [(list(range(10)), 6), ([10, 11], 2)]
    _check(*_shared_case(lens, groups, dtype, Hq, Hk, D, B, seed=93), num_ctas=11)


@pytest.mark.parametrize("dtype,Hq,Hk,D", [("f32", 8, 2, 128), ("f16", 4, 4, 64)])
def test_prefix_aware_plain_fallback(dtype, Hq, Hk, D):
    # shapes outside the one-launch variants (fp32; one q head of 64
    # elements per kv head) are decoded by the plain decode
    lens, groups = _two_groups()
    _check(*_shared_case(lens, groups, dtype, Hq, Hk, D, seed=94),
           tol=1e-5 if dtype == "f32" else 2e-3)


def test_prefix_aware_counters_return_to_zero():
    lens, groups = _two_groups()
    q, kp, vp, bt, cl, gos, gpb = _shared_case(lens, groups)
    n = binding.prefix_workspace_bytes(kp, len(lens), 32, bt.shape[1], gos, gpb)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    for _ in range(3):             # one workspace, calls in a row
        _check(q, kp, vp, bt, cl, gos, gpb, workspace=ws, num_ctas=9)
    assert int((ws[: 4096 * 16] != 0).sum()) == 0        # split-K arrival counters
    # the (sequence, kv head, merge slice) counters close the workspace (a
    # 256-byte-aligned region of 7 x 8 x 4 counters)
    assert int((ws[-1024:] != 0).sum()) == 0


def test_prefix_aware_lse_out():
    lens, groups = _two_groups()
    q, kp, vp, bt, cl, gos, gpb = _shared_case(lens, groups)
    lse = torch.empty(len(lens), 32, dtype=torch.float32, device="cuda")
    _check(q, kp, vp, bt, cl, gos, gpb, lse_out=lse)
    ref = torch.empty_like(lse)
    binding.decode_attention(q.cuda(), kp.cuda(), vp.cuda(), bt.cuda(), cl.cuda(),
                             1.0 / math.sqrt(128), out_dtype=torch.float32, lse_out=ref)
    torch.cuda.synchronize()
    assert float((lse - ref).abs().max()) < 1e-4


@pytest.mark.parametrize("suffix_hi", [28000, 500])
def test_prefix_aware_on_the_shared_prefix_workload(suffix_hi):
    # the 20-agent workload (4000-token shared prefix, copy-on-write of its
    # last block), with its suffixes and with short ones; every output element
    spec = W.SPECS[3].__class__(**{**W.SPECS[3].__dict__, "suffix_hi": suffix_hi})
    st, vals = W.make_workload(spec, seed=0)
    kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
    oracle.block_copy(st.cow_pairs, kp, vp)
    oracle.append(vals["k_new"], vals["v_new"], st.slot_mapping, kp, vp)
    pb = spec.shared_prefix // spec.block_size
    # after the copy-on-write the last prefix block is private to all but one
    # holder, so the group shares the blocks before it
    gos, gpb = [0] * st.context_lens.numel(), [pb - 1]
    _check(vals["q"], kp, vp, st.block_tables, st.context_lens, gos, gpb)


def test_lse_out_is_log2_of_the_softmax_denominator():
    spec = W.WorkloadSpec("lse", 4, 8, 2, 64, 16, "f16", 1.0)
    st, vals = W.make_workload(spec, seed=92, lengths=[1, 70, 0, 300])
    kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
    oracle.append(vals["k_new"], vals["v_new"], st.slot_mapping, kp, vp)
    scale = 0.2
    lse = torch.empty(4, 8, dtype=torch.float32, device="cuda")
    binding.decode_attention(vals["q"].cuda(), kp.cuda(), vp.cuda(), st.block_tables.cuda(),
                             st.context_lens.cuda(), scale, out_dtype=torch.float32,
                             num_ctas=5, lse_out=lse)
    torch.cuda.synchronize()
    got = lse.cpu().double().numpy()
    B = 16
    for s, L in enumerate(st.context_lens.tolist()):
        for h in range(8):
            if L == 0:
                assert got[s, h] == -np.inf
                continue
            g = h // 4
            rows = [kp[int(st.block_tables[s, t // B]), g, t % B].double().numpy() for t in range(L)]
            z = scale * np.array(rows) @ vals["q"][s, h].double().numpy()
            want = (np.log(np.sum(np.exp(z - z.max()))) + z.max()) / np.log(2.0)
            assert abs(got[s, h] - want) < 1e-4, (s, h)


def test_prefix_groups_are_checked():
    lens, groups = _two_groups()
    q, kp, vp, bt, cl, gos, gpb = _shared_case(lens, groups)
    q, kp, vp = q.cuda(), kp.cuda(), vp.cuda()
    with pytest.raises(binding.PkvError):
        binding.decode_attention_prefix(q, kp, vp, bt.cuda(), cl.cuda(), 0.1, [0] * 7, [0])
    with pytest.raises(binding.PkvError):
        binding.decode_attention_prefix(q, kp, vp, bt.cuda(), cl.cuda(), 0.1, [3] * 7, [2])
