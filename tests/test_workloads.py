"""Structure checks for the seeded workload generator (CPU only)."""
import math

import torch

from paged_kv_cache_47_gb300 import workloads as W


def _blocks(st, s):
    L = int(st.context_lens[s])
    B = st.spec.block_size
    return st.block_tables[s, : -(-L // B)].tolist()


def test_specs_match_the_five_workloads():
    s = W.SPECS
    assert (s[0].num_seqs, s[0].num_q_heads, s[0].num_kv_heads, s[0].head_dim, s[0].dtype) == (4, 4, 4, 64, "f32")
    assert (s[1].num_seqs, s[1].num_q_heads, s[1].num_kv_heads, s[1].head_dim, s[1].dtype) == (64, 32, 8, 128, "bf16")
    assert (s[2].num_seqs, s[2].num_q_heads, s[2].num_kv_heads, s[2].std) == (256, 40, 40, 0.5)
    assert (s[3].num_seqs, s[3].shared_prefix, s[3].suffix_hi, s[3].cow) == (20, 4000, 28000, True)
    assert (s[4].num_seqs, s[4].num_q_heads, s[4].num_kv_heads, s[4].len_lo, s[4].len_hi) == (8, 64, 8, 32768, 131072)


def test_private_tables_are_disjoint_and_sized():
    st = W.make_structure(W.SPECS[1], seed=0)
    L = st.context_lens
    assert int(L.min()) >= 512 and int(L.max()) <= 4096
    seen = set()
    for s in range(L.numel()):
        b = _blocks(st, s)
        assert not (seen & set(b))
        seen |= set(b)
        assert all(0 <= x < st.num_blocks for x in b)
    need = sum(-(-int(x) // 16) for x in L)
    assert st.num_blocks == math.ceil(1.2 * need)


def test_slot_mapping_points_at_last_token():
    st = W.make_structure(W.SPECS[2], seed=0)
    B = st.spec.block_size
    for s in range(st.context_lens.numel()):
        p = int(st.context_lens[s]) - 1
        assert int(st.slot_mapping[s]) == int(st.block_tables[s, p // B]) * B + p % B


def test_prefix_sharing_and_copy_on_write():
    st = W.make_structure(W.SPECS[3], seed=0)
    S, B = 20, 16
    pre = st.block_tables_pre_cow
    for s in range(1, S):
        assert torch.equal(pre[s, :250], pre[0, :250])          # shared prefix ids
    pairs = st.cow_pairs
    assert pairs.shape == (S - 1, 2)                              # last holder keeps it
    assert torch.all(pairs[:, 0] == pre[0, 249])
    assert len(set(pairs[:, 1].tolist())) == S - 1
    post = st.block_tables
    assert len(set(post[:, 249].tolist())) == S                  # every writer private
    for s in range(S):
        assert torch.equal(post[s, :249], pre[s, :249])


def test_nan_sentinels_cover_tails_and_append_slot():
    spec = W.WorkloadSpec("t", 3, 2, 1, 8, 4, "f32", 1.0, 1, 1)
    st, v = W.make_workload(spec, lengths=[5, 8, 1])
    kp = v["k_pool"]
    t = st.block_tables
    assert torch.isnan(kp[t[0, 1], 0, 0:4]).all()       # L=5: slot 4 (pre-append) and tail
    assert not torch.isnan(kp[t[0, 0]]).any()
    assert torch.isnan(kp[t[1, 1], 0, 3]).all()         # L=8: pre-append slot
    assert not torch.isnan(kp[t[1, 1], 0, :3]).any()
    assert torch.isnan(kp[t[2, 0], 0, :]).all()         # L=1
    used = set(t[t >= 0].tolist())
    for b in range(st.num_blocks):
        if b not in used:
            assert torch.isnan(kp[b]).all()


def test_seeded_and_reproducible():
    a = W.make_structure(W.SPECS[4], seed=0)
    b = W.make_structure(W.SPECS[4], seed=0)
    c = W.make_structure(W.SPECS[4], seed=1)
    assert torch.equal(a.block_tables, b.block_tables)
    assert not torch.equal(a.context_lens, c.context_lens)
