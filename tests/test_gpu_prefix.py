"""Prefix-aware decode (pkv_decode_attention_prefix) and the decode's lse_out
option, against the oracle.

The prefix-aware call must give the plain decode's result (the oracle's
dense attention over each whole context) within 2e-3, for groups of
sequences that share leading blocks, sequences in no group, and members whose
private suffix is empty. lse_out must be log2 of each head's softmax
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


def _two_prefix_case(dtype="bf16", Hq=32, Hk=8, B=16, seed=91):
    """Sequences 0-3 share a 5-block prefix, 4-5 share a 3-block prefix,
    6 is on its own; tables built here, values drawn by the generator."""
    lens = [5 * B + 30, 5 * B + 200, 5 * B, 5 * B + 1, 3 * B + 77, 3 * B + 5, 400]
    spec = W.WorkloadSpec("pfx", len(lens), Hq, Hk, 128, B, dtype, 1.0, pool_ratio=1.0)
    st, vals = W.make_workload(spec, seed=seed, lengths=lens)
    bt = st.block_tables.clone()
    bt[1:4, :5] = bt[0, :5]                       # group 0 shares sequence 0's first 5 blocks
    bt[5, :3] = bt[4, :3]                         # group 1 shares sequence 4's first 3 blocks
    return st, vals, bt, torch.tensor(lens, dtype=torch.int32), [0, 0, 0, 0, 1, 1, -1], [5, 3]


@pytest.mark.parametrize("num_ctas", [0, 7])
def test_prefix_aware_equals_plain_decode(num_ctas):
    st, vals, bt, cl, gos, gpb = _two_prefix_case()
    kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
    oracle.append(vals["k_new"], vals["v_new"], st.slot_mapping, kp, vp)
    scale = 1.0 / math.sqrt(128)
    want = oracle.decode(vals["q"], kp, vp, bt, cl, scale)
    out = binding.decode_attention_prefix(vals["q"].cuda(), kp.cuda(), vp.cuda(), bt.cuda(),
                                          cl.cuda(), scale, gos, gpb, out_dtype=torch.float32,
                                          num_ctas=num_ctas)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert binding.get_error() == 0
    assert np.all(np.isfinite(got)) and float(np.max(np.abs(got - want))) <= 2e-3


def test_prefix_aware_on_the_shared_prefix_workload_sampled():
    st, vals = W.make_workload(3, seed=0)
    kp, vp = vals["k_pool"].clone(), vals["v_pool"].clone()
    oracle.block_copy(st.cow_pairs, kp, vp)
    oracle.append(vals["k_new"], vals["v_new"], st.slot_mapping, kp, vp)
    spec = W.SPECS[3]
    pb = spec.shared_prefix // spec.block_size
    # after the copy-on-write the last prefix block is private to all but one
    # holder, so the group shares the blocks before it
    gos, gpb = [0] * st.context_lens.numel(), [pb - 1]
    scale = 1.0 / math.sqrt(spec.head_dim)
    out = binding.decode_attention_prefix(vals["q"].cuda(), kp.cuda(), vp.cuda(),
                                          st.block_tables.cuda(), st.context_lens.cuda(), scale,
                                          gos, gpb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    ids = [0, 7, 19]
    want = oracle.decode(vals["q"], kp, vp, st.block_tables, st.context_lens, scale, seq_ids=ids)
    got = out.double().cpu().numpy()[ids]
    assert float(np.max(np.abs(got - want))) <= 2e-3


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
    st, vals, bt, cl, gos, gpb = _two_prefix_case()
    q, kp, vp = vals["q"].cuda(), vals["k_pool"].cuda(), vals["v_pool"].cuda()
    with pytest.raises(binding.PkvError):
        binding.decode_attention_prefix(q, kp, vp, bt.cuda(), cl.cuda(), 0.1, [0] * 7, [0])
    with pytest.raises(binding.PkvError):
        binding.decode_attention_prefix(q, kp, vp, bt.cuda(), cl.cuda(), 0.1, [3] * 7, [2])
