"""Pins for the CPU oracle: each test fixes the oracle to something other than
itself — a library routine, a closed form, an invariant the pages state, an
exhaustive decode check, or a value printed on the pages.

A plausible mistake anywhere in the oracle (dropped scale, wrong GQA head map,
wrong token offset in a block, transposed operand, missing max subtraction,
wrong fp16/bf16 decode, reading past a context length) fails at least one of
these.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


# --------------------------------------------------------------------------
# helpers: the tests build paged pools from dense K/V with their own scatter
# --------------------------------------------------------------------------
def _page(dense_k, dense_v, B, NB, gen, nan_fill=True):
    """Scatter dense per-sequence K/V ([L][Hk][D] each) into a pool [NB][Hk][B][D]
    at a random permutation of physical blocks. Returns pools, tables, lens."""
    S = len(dense_k)
    Hk, D = dense_k[0].shape[1], dense_k[0].shape[2]
    dt = dense_k[0].dtype
    need = sum(-(-k.shape[0] // B) for k in dense_k)
    assert need <= NB
    perm = torch.randperm(NB, generator=gen)
    fill = float("nan") if nan_fill else 0.0
    kp = torch.full((NB, Hk, B, D), fill, dtype=dt)
    vp = torch.full((NB, Hk, B, D), fill, dtype=dt)
    M = max(1, max(-(-k.shape[0] // B) for k in dense_k))
    tables = torch.full((S, M), -1, dtype=torch.int32)
    c = 0
    for s in range(S):
        L = dense_k[s].shape[0]
        for j in range(-(-L // B)):
            phys = int(perm[c]); c += 1
            tables[s, j] = phys
            n = min(B, L - j * B)
            kp[phys, :, :n, :] = dense_k[s][j * B:j * B + n].transpose(0, 1)
            vp[phys, :, :n, :] = dense_v[s][j * B:j * B + n].transpose(0, 1)
    lens = torch.tensor([k.shape[0] for k in dense_k], dtype=torch.int32)
    return kp, vp, tables, lens


def _sdpa(q, dense_k, dense_v, scale):
    """Reference: torch SDPA in fp64 on contiguous K/V; GQA by repeat_interleave."""
    S, Hq, D = q.shape
    out = np.zeros((S, Hq, D))
    for s in range(S):
        K = dense_k[s].to(torch.float64).transpose(0, 1)  # [Hk][L][D]
        V = dense_v[s].to(torch.float64).transpose(0, 1)
        G = Hq // K.shape[0]
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        qq = q[s].to(torch.float64).unsqueeze(1)           # [Hq][1][D]
        o = torch.nn.functional.scaled_dot_product_attention(qq, K, V, scale=scale)
        out[s] = o[:, 0, :].numpy()
    return out


def _rand_case(S, Hq, Hk, D, B, dtype, lens, seed, std=1.0, slack=3):
    g = torch.Generator().manual_seed(seed)
    dt = DT[dtype]
    dk = [(torch.randn(L, Hk, D, generator=g) * std).to(dt) for L in lens]
    dv = [(torch.randn(L, Hk, D, generator=g) * std).to(dt) for L in lens]
    q = (torch.randn(S, Hq, D, generator=g) * std).to(dt)
    need = sum(-(-L // B) for L in lens)
    kp, vp, bt, cl = _page(dk, dv, B, need + slack, g)
    return q, dk, dv, kp, vp, bt, cl


# --------------------------------------------------------------------------
# element decoding
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decoder_exhaustive_16bit(dtype):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32)
    ref = bits.to(torch.int16).view(DT[dtype]).to(torch.float64).numpy()
    got = np.array([oracle.decode_elem(DT[dtype], int(b)) for b in bits.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_decoder_f32_sampled():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(-(1 << 31), (1 << 31) - 1, (20000,), generator=g, dtype=torch.int64)
    specials = torch.tensor([0, 1, 0x7F800000, 0xFF800000 - (1 << 32), 0x00800000, 0x3F800000],
                            dtype=torch.int64)
    bits = torch.cat([bits, specials]).to(torch.int32)
    ref = bits.view(torch.float32).to(torch.float64).numpy()
    got = np.array([oracle.decode_elem(torch.float32, int(b) & 0xFFFFFFFF) for b in bits.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


# --------------------------------------------------------------------------
# decode vs a library routine on the contiguous layout
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("Hq,Hk,D,B", [(4, 4, 16, 4), (8, 2, 32, 8), (8, 1, 16, 16), (6, 3, 8, 4)])
def test_decode_matches_sdpa_on_contiguous(dtype, Hq, Hk, D, B):
    lens = [1, 5, B, B + 1, 3 * B - 1, 37]
    q, dk, dv, kp, vp, bt, cl = _rand_case(len(lens), Hq, Hk, D, B, dtype, lens, seed=11)
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode(q, kp, vp, bt, cl, scale)
    ref = _sdpa(q, dk, dv, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_decode_scale_is_applied():
    lens = [9, 20]
    q, dk, dv, kp, vp, bt, cl = _rand_case(2, 4, 2, 16, 4, "f32", lens, seed=5)
    for scale in (0.05, 0.7, 3.0):
        np.testing.assert_allclose(oracle.decode(q, kp, vp, bt, cl, scale),
                                   _sdpa(q, dk, dv, scale), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# closed forms and special cases
# --------------------------------------------------------------------------
def test_single_token_context_returns_its_v():
    q, dk, dv, kp, vp, bt, cl = _rand_case(3, 8, 2, 32, 16, "bf16", [1, 1, 1], seed=7)
    got = oracle.decode(q, kp, vp, bt, cl, 0.125)
    for s in range(3):
        for h in range(8):
            assert np.array_equal(got[s, h], dv[s][0, h // 4].to(torch.float64).numpy())


def test_constant_v_returns_that_v():
    g = torch.Generator().manual_seed(8)
    lens = [1, 17, 64]
    Hk, D = 2, 16
    c = (torch.randn(Hk, D, generator=g)).to(torch.bfloat16)
    dk = [torch.randn(L, Hk, D, generator=g).to(torch.bfloat16) for L in lens]
    dv = [c.unsqueeze(0).expand(L, Hk, D).clone() for L in lens]
    q = torch.randn(3, 4, D, generator=g).to(torch.bfloat16)
    kp, vp, bt, cl = _page(dk, dv, 8, 20, g)
    got = oracle.decode(q, kp, vp, bt, cl, 0.25)
    for s in range(3):
        for h in range(4):
            np.testing.assert_allclose(got[s, h], c[h // 2].double().numpy(), rtol=1e-15, atol=0)


def test_zero_query_gives_mean_of_v():
    lens = [3, 33]
    q, dk, dv, kp, vp, bt, cl = _rand_case(2, 4, 4, 16, 8, "f16", lens, seed=9)
    q.zero_()
    got = oracle.decode(q, kp, vp, bt, cl, 0.25)
    for s in range(2):
        mean = dv[s].to(torch.float64).mean(dim=0).numpy()   # [Hk][D]
        np.testing.assert_allclose(got[s], mean, rtol=1e-13, atol=1e-15)


def test_two_token_logistic_closed_form():
    q, dk, dv, kp, vp, bt, cl = _rand_case(1, 2, 1, 8, 4, "f32", [2], seed=13)
    scale = 0.9
    got = oracle.decode(q, kp, vp, bt, cl, scale)
    K = dk[0][:, 0].double().numpy(); V = dv[0][:, 0].double().numpy()
    for h in range(2):
        qq = q[0, h].double().numpy()
        z0, z1 = scale * qq @ K[0], scale * qq @ K[1]
        a = 1.0 / (1.0 + math.exp(z1 - z0))        # logistic(z0 - z1)
        ref = a * V[0] + (1.0 - a) * V[1]
        np.testing.assert_allclose(got[0, h], ref, rtol=1e-13, atol=1e-15)


def test_large_logits_no_overflow_hard_attention():
    # logits ~1e5: exp without max subtraction overflows; the argmax token wins.
    g = torch.Generator().manual_seed(21)
    L, D = 40, 16
    dk = [torch.randn(L, 1, D, generator=g)]
    dv = [torch.randn(L, 1, D, generator=g)]
    q = dk[0][23, 0].clone().view(1, 1, D) * 3.0
    kp, vp, bt, cl = _page(dk, dv, 8, 8, g)
    got = oracle.decode(q, kp, vp, bt, cl, 1e4)
    scores = (dk[0][:, 0].double() @ q[0, 0].double())
    assert int(scores.argmax()) == 23
    assert np.all(np.isfinite(got))
    assert np.array_equal(got[0, 0], dv[0][23, 0].double().numpy())


def test_gqa_head_mapping():
    # kv head g holds constant V = g + 1: q head h must read kv head h // G
    g = torch.Generator().manual_seed(4)
    Hq, Hk, D, L = 12, 3, 8, 19
    dk = [torch.randn(L, Hk, D, generator=g)]
    dv = [torch.arange(1, Hk + 1, dtype=torch.float32).view(1, Hk, 1).expand(L, Hk, D).clone()]
    q = torch.randn(1, Hq, D, generator=g)
    kp, vp, bt, cl = _page(dk, dv, 4, 6, g)
    got = oracle.decode(q, kp, vp, bt, cl, 0.3)
    for h in range(Hq):
        np.testing.assert_allclose(got[0, h], np.full(D, h // (Hq // Hk) + 1.0), rtol=1e-15)


def test_context_len_zero_gives_zeros():
    q, dk, dv, kp, vp, bt, cl = _rand_case(2, 4, 2, 8, 4, "f32", [5, 7], seed=1)
    cl[1] = 0
    got = oracle.decode(q, kp, vp, bt, cl, 0.5)
    assert np.array_equal(got[1], np.zeros_like(got[1]))


def test_out_of_range_block_is_an_error():
    q, dk, dv, kp, vp, bt, cl = _rand_case(1, 2, 2, 8, 4, "f32", [9], seed=2)
    bt[0, 1] = kp.shape[0]
    with pytest.raises(ValueError):
        oracle.decode(q, kp, vp, bt, cl, 0.5)


# --------------------------------------------------------------------------
# invariants the pages state
# --------------------------------------------------------------------------
def test_permuted_physical_layout_is_invisible():
    # "the program never knows" where its pages live: two random layouts of the
    # same dense data give bit-identical results
    g = torch.Generator().manual_seed(31)
    lens = [50, 7, 33]
    dk = [torch.randn(L, 2, 16, generator=g).to(torch.bfloat16) for L in lens]
    dv = [torch.randn(L, 2, 16, generator=g).to(torch.bfloat16) for L in lens]
    q = torch.randn(3, 8, 16, generator=g).to(torch.bfloat16)
    a = _page(dk, dv, 8, 40, torch.Generator().manual_seed(1))
    b = _page(dk, dv, 8, 40, torch.Generator().manual_seed(2))
    assert not torch.equal(a[2], b[2])
    ra = oracle.decode(q, a[0], a[1], a[2], a[3], 0.25)
    rb = oracle.decode(q, b[0], b[1], b[2], b[3], 0.25)
    assert np.array_equal(ra, rb)


def test_tail_and_unused_blocks_are_never_read():
    g = torch.Generator().manual_seed(6)
    lens = [13, 3]
    dk = [torch.randn(L, 1, 8, generator=g) for L in lens]
    dv = [torch.randn(L, 1, 8, generator=g) for L in lens]
    q = torch.randn(2, 1, 8, generator=g)
    kp, vp, bt, cl = _page(dk, dv, 8, 10, torch.Generator().manual_seed(0), nan_fill=True)
    kz, vz, bz, cz = _page(dk, dv, 8, 10, torch.Generator().manual_seed(0), nan_fill=False)
    ra = oracle.decode(q, kp, vp, bt, cl, 0.4)
    rb = oracle.decode(q, kz, vz, bz, cz, 0.4)
    assert np.all(np.isfinite(ra)) and np.array_equal(ra, rb)


def test_shared_prefix_equals_private_copies():
    # sequences whose tables point at the same physical prefix blocks give the
    # same result as sequences holding private copies of those blocks
    g = torch.Generator().manual_seed(12)
    B, Hk, D, P = 8, 2, 16, 24
    prefix_k = torch.randn(P, Hk, D, generator=g).to(torch.float16)
    prefix_v = torch.randn(P, Hk, D, generator=g).to(torch.float16)
    suf = [5, 0, 19]
    dk = [torch.cat([prefix_k, torch.randn(n, Hk, D, generator=g).to(torch.float16)]) for n in suf]
    dv = [torch.cat([prefix_v, torch.randn(n, Hk, D, generator=g).to(torch.float16)]) for n in suf]
    q = torch.randn(3, 4, D, generator=g).to(torch.float16)
    kp, vp, bt, cl = _page(dk, dv, B, 30, torch.Generator().manual_seed(3))
    private = oracle.decode(q, kp, vp, bt, cl, 0.25)
    # repoint every sequence's prefix entries at sequence 0's physical blocks
    bt2 = bt.clone()
    for s in range(1, 3):
        bt2[s, :P // B] = bt[0, :P // B]
    kp2, vp2 = kp.clone(), vp.clone()
    for s in range(1, 3):                     # the private copies are now dead
        kp2[bt[s, :P // B].long()] = float("nan")
        vp2[bt[s, :P // B].long()] = float("nan")
    shared = oracle.decode(q, kp2, vp2, bt2, cl, 0.25)
    assert np.array_equal(private, shared)


def test_copy_on_write_leaves_output_unchanged():
    g = torch.Generator().manual_seed(14)
    lens = [20, 20]
    dk = [torch.randn(20, 2, 8, generator=g)] * 2
    dv = [torch.randn(20, 2, 8, generator=g)] * 2
    q = torch.randn(2, 2, 8, generator=g)
    kp, vp, bt, cl = _page(dk, dv, 8, 12, torch.Generator().manual_seed(5))
    bt[1, :] = bt[0, :]                            # sequence 1 shares all of 0's blocks
    before = oracle.decode(q, kp, vp, bt, cl, 0.5)
    used = set(bt[0].tolist())
    fresh = next(b for b in range(12) if b not in used)
    oracle.block_copy([[int(bt[0, 1]), fresh]], kp, vp)
    bt[1, 1] = fresh
    after = oracle.decode(q, kp, vp, bt, cl, 0.5)
    assert np.array_equal(before, after)


# --------------------------------------------------------------------------
# the page's example block table
# --------------------------------------------------------------------------
def test_block_table_example_from_page():
    ex = json.load(open(os.path.join(GOLDEN, "block_table_example.json")))
    B = ex["block_size"]
    sessions = ex["sessions"]
    NB, D = 100, 8
    # V row at (phys, off) encodes its own address; K rows are zero except the
    # target token, so hard attention returns the V row the table walk reaches
    vp = torch.zeros(NB, 1, B, D)
    for p in range(NB):
        for o in range(B):
            vp[p, 0, o, :] = p * 100 + o
    names = sorted(sessions)
    M = max(len(sessions[n]) for n in names)
    bt = torch.full((len(names), M), -1, dtype=torch.int32)
    for i, n in enumerate(names):
        bt[i, :len(sessions[n])] = torch.tensor(sessions[n], dtype=torch.int32)
    cl = torch.tensor([len(sessions[n]) * B for n in names], dtype=torch.int32)
    for i, n in enumerate(names):
        for t in range(0, int(cl[i]), 5):
            kp = torch.zeros(NB, 1, B, D)
            phys, off = sessions[n][t // B], t % B
            kp[phys, 0, off, :] = 1.0
            q = torch.zeros(len(names), 1, D)
            q[i, 0, :] = 1.0
            out = oracle.decode(q, kp, vp, bt, cl, 1e3)
            assert out[i, 0, 0] == phys * 100 + off, (n, t)


# --------------------------------------------------------------------------
# append and block copy against plain tensor indexing
# --------------------------------------------------------------------------
def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_append_matches_indexed_assignment(dtype):
    g = torch.Generator().manual_seed(17)
    NB, Hk, B, D, N = 9, 3, 8, 16, 7
    dt = DT[dtype]
    kp = torch.randn(NB, Hk, B, D, generator=g).to(dt)
    vp = torch.randn(NB, Hk, B, D, generator=g).to(dt)
    kn = torch.randn(N, Hk, D, generator=g).to(dt)
    vn = torch.randn(N, Hk, D, generator=g).to(dt)
    slots = torch.randperm(NB * B, generator=g)[:N].to(torch.int64)
    slots[2] = -1                                   # negative slot: skipped
    ek, ev = kp.clone(), vp.clone()
    keep = slots >= 0
    s = slots[keep]
    ek[s // B, :, s % B, :] = kn[keep]
    ev[s // B, :, s % B, :] = vn[keep]
    oracle.append(kn, vn, slots, kp, vp)
    assert torch.equal(_bits(kp), _bits(ek)) and torch.equal(_bits(vp), _bits(ev))


def test_append_out_of_range_slot_is_an_error():
    kp = torch.zeros(2, 1, 4, 4); vp = torch.zeros(2, 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.append(torch.zeros(1, 1, 4), torch.zeros(1, 1, 4), torch.tensor([8]), kp, vp)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_block_copy_matches_indexed_copy(dtype):
    g = torch.Generator().manual_seed(19)
    NB, Hk, B, D = 12, 2, 16, 8
    dt = DT[dtype]
    kp = torch.randn(NB, Hk, B, D, generator=g).to(dt)
    vp = torch.randn(NB, Hk, B, D, generator=g).to(dt)
    pairs = [[3, 7], [0, 11], [5, 1]]
    ek, ev = kp.clone(), vp.clone()
    for a, b in pairs:
        ek[b] = ek[a]
        ev[b] = ev[a]
    oracle.block_copy(pairs, kp, vp)
    assert torch.equal(_bits(kp), _bits(ek)) and torch.equal(_bits(vp), _bits(ev))
