"""Pins of the flat-span decode oracle (one contiguous, token-major span per
sequence instead of blocks; "Contiguous vs Paged KV Cache on RDNA4", section
"Why the single-user verdict flipped": the kernel reads a flat span and the
result does not change).

- Equal to the paged oracle on the same rows laid out in shuffled blocks.
- Equal to torch's scaled_dot_product_attention in fp64.
- Zero length gives zeros; a bad slot or a length past the capacity is an error.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle


def _case(dtype, S, Hq, Hk, D, cap, lens, seed, num_slots=None):
    g = torch.Generator().manual_seed(seed)
    NS = num_slots or S + 2
    kf = torch.randn(NS, cap, Hk, D, generator=g).to(dtype)
    vf = torch.randn(NS, cap, Hk, D, generator=g).to(dtype)
    q = torch.randn(S, Hq, D, generator=g).to(dtype)
    slots = torch.randperm(NS, generator=g)[:S].to(torch.int32)
    return q, kf, vf, slots, torch.tensor(lens, dtype=torch.int32)


@pytest.mark.parametrize("dtype,Hq,Hk,B", [(torch.bfloat16, 8, 2, 16), (torch.float16, 4, 4, 8),
                                           (torch.float32, 6, 3, 32)])
def test_flat_equals_paged_on_the_same_rows(dtype, Hq, Hk, B):
    S, D, cap = 4, 64, 96
    lens = [1, 17, 64, 96]
    q, kf, vf, slots, cl = _case(dtype, S, Hq, Hk, D, cap, lens, seed=71)
    # the same rows, cut into blocks of B tokens placed at shuffled block ids
    nblk = [(L + B - 1) // B for L in lens]
    NB = sum(nblk) + 2
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(72))
    kp = torch.zeros(NB, Hk, B, D, dtype=dtype)
    vp = torch.zeros_like(kp)
    tables = torch.full((S, max(nblk)), -1, dtype=torch.int32)
    k = 0
    for s, L in enumerate(lens):
        for j in range(nblk[s]):
            b = int(perm[k])
            k += 1
            tables[s, j] = b
            for o in range(B):
                t = j * B + o
                if t < L:
                    kp[b, :, o] = kf[slots[s], t]
                    vp[b, :, o] = vf[slots[s], t]
    scale = 1.0 / math.sqrt(D)
    flat = oracle.decode_flat(q, kf, vf, slots, cl, scale)
    paged = oracle.decode(q, kp, vp, tables, cl, scale)
    assert np.array_equal(flat, paged)


def test_flat_equals_sdpa():
    S, Hq, Hk, D, cap = 3, 8, 4, 32, 50
    lens = [5, 50, 23]
    q, kf, vf, slots, cl = _case(torch.bfloat16, S, Hq, Hk, D, cap, lens, seed=73)
    scale = 0.3
    got = oracle.decode_flat(q, kf, vf, slots, cl, scale)
    for s, L in enumerate(lens):
        K = kf[slots[s], :L].to(torch.float64).permute(1, 0, 2)     # [Hk][L][D]
        V = vf[slots[s], :L].to(torch.float64).permute(1, 0, 2)
        K, V = K.repeat_interleave(Hq // Hk, 0), V.repeat_interleave(Hq // Hk, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[s].to(torch.float64).unsqueeze(1), K, V, scale=scale).squeeze(1)
        assert np.max(np.abs(got[s] - ref.numpy())) < 1e-12


def test_flat_zero_length_and_errors():
    q, kf, vf, slots, cl = _case(torch.float16, 2, 4, 2, 16, 8, [0, 3], seed=74)
    out = oracle.decode_flat(q, kf, vf, slots, cl, 1.0)
    assert np.all(out[0] == 0) and np.all(np.isfinite(out[1]))
    with pytest.raises(ValueError):
        oracle.decode_flat(q, kf, vf, torch.tensor([0, 99], dtype=torch.int32), cl, 1.0)
    with pytest.raises(ValueError):
        oracle.decode_flat(q, kf, vf, slots, torch.tensor([0, 9], dtype=torch.int32), 1.0)
