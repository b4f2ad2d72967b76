"""Flat spans (pkv_flat_*: a KV cache contiguous in virtual memory, physical
chunks mapped on demand) against the flat-span oracle, and against the paged
path on the same rows.

- Decode over flat spans matches oracle_decode_flat within 2e-3.
- On the same rows, flat and paged decodes are bitwise equal: the kernel's
  decomposition and arithmetic are the same, only the addressing differs.
- Growing a slot keeps what it holds; a released slot is never read (its
  length is clamped to zero with PKV_DEVERR_CONTEXT); appends past the
  committed tokens or to a bad slot are refused with PKV_DEVERR_SLOT.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_cache_47_gb300 import binding, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


def make_flat(dtype, NS, cap, Hk, D, lens, seed):
    """A flat cache whose slot i holds lens[i] random rows (lens[i] may be 0),
    and the same rows on the host [NS][cap][Hk][D]."""
    g = torch.Generator().manual_seed(seed)
    fc = binding.FlatCache(NS, cap, Hk, D, dtype)
    hk = torch.full((NS, cap, Hk, D), float("nan")).to(dtype)
    hv = hk.clone()
    for slot, L in enumerate(lens):
        if L == 0:
            continue
        fc.reserve(slot, L)
        k = torch.randn(L, Hk, D, generator=g).to(dtype)
        v = torch.randn(L, Hk, D, generator=g).to(dtype)
        hk[slot, :L], hv[slot, :L] = k, v
        sl = torch.full((L,), slot, dtype=torch.int32, device="cuda")
        pos = torch.arange(L, dtype=torch.int32, device="cuda")
        fc.append(k.cuda(), v.cuda(), sl, pos)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    return fc, hk, hv


@pytest.mark.parametrize("dtype,Hq,Hk,D", [(torch.bfloat16, 32, 8, 128), (torch.float16, 8, 8, 128),
                                           (torch.bfloat16, 16, 2, 64), (torch.float16, 40, 2, 128)])
@pytest.mark.parametrize("num_ctas", [0, 5])
def test_flat_decode_matches_oracle(dtype, Hq, Hk, D, num_ctas):
    lens = [1, 63, 64, 65, 300, 1000, 0, 129]
    fc, hk, hv = make_flat(dtype, len(lens) + 1, 1024, Hk, D, lens, seed=81)
    g = torch.Generator().manual_seed(82)
    order = [5, 0, 7, 2, 6, 4, 1, 3]                 # batch entries in any slot order
    slots = torch.tensor(order, dtype=torch.int32)
    cl = torch.tensor([lens[i] for i in order], dtype=torch.int32)
    q = torch.randn(len(order), Hq, D, generator=g).to(dtype)
    scale = 1.0 / math.sqrt(D)
    out = fc.decode_attention(q.cuda(), slots.cuda(), cl.cuda(), scale, out_dtype=torch.float32,
                              num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    want = oracle.decode_flat(q, hk, hv, slots, cl, scale)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got)) and float(np.max(np.abs(got - want))) <= 2e-3
    fc.close()


def test_flat_and_paged_are_bitwise_equal():
    dtype, Hq, Hk, D, B = torch.bfloat16, 32, 8, 128, 16
    lens = [700, 64, 1, 2049, 333]
    fc, hk, hv = make_flat(dtype, len(lens), 2112, Hk, D, lens, seed=83)
    # the same rows in a paged pool, blocks at shuffled ids
    nblk = [(L + B - 1) // B for L in lens]
    NB = sum(nblk) + 5
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(84))
    kp = torch.zeros(NB, Hk, B, D, dtype=dtype)
    vp = torch.zeros_like(kp)
    tables = torch.full((len(lens), max(nblk)), -1, dtype=torch.int32)
    k = 0
    for s, L in enumerate(lens):
        for j in range(nblk[s]):
            b = int(perm[k])
            k += 1
            tables[s, j] = b
            n = min(B, L - j * B)
            kp[b, :, :n] = hk[s, j * B:j * B + n].transpose(0, 1)
            vp[b, :, :n] = hv[s, j * B:j * B + n].transpose(0, 1)
    q = torch.randn(len(lens), Hq, D, generator=torch.Generator().manual_seed(85)).to(dtype).cuda()
    cl = torch.tensor(lens, dtype=torch.int32).cuda()
    slots = torch.arange(len(lens), dtype=torch.int32).cuda()
    scale = 1.0 / math.sqrt(D)
    for C in (0, 7, 300):
        flat = fc.decode_attention(q, slots, cl, scale, out_dtype=torch.float32, num_ctas=C)
        paged = binding.decode_attention(q, kp.cuda(), vp.cuda(), tables.cuda(), cl, scale,
                                         out_dtype=torch.float32, num_ctas=C)
        torch.cuda.synchronize()
        assert torch.equal(flat, paged), C
    assert binding.get_error() == 0
    fc.close()


def test_flat_tables_ready_matches_default():
    dtype, Hq, Hk, D = torch.bfloat16, 32, 8, 128
    lens = [0, 500, 64, 1300]
    fc, hk, hv = make_flat(dtype, len(lens), 2048, Hk, D, lens, seed=88)
    g = torch.Generator().manual_seed(89)
    q = torch.randn(len(lens), Hq, D, generator=g).to(dtype).cuda()
    kn = torch.randn(len(lens), Hk, D, generator=g).to(dtype).cuda()
    slots = torch.arange(len(lens), dtype=torch.int32, device="cuda")
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    # rewrite each sequence's last row (flat append), then decode, three times
    live = [i for i, L in enumerate(lens) if L > 0]
    sl = torch.tensor(live, dtype=torch.int32, device="cuda")
    pos = torch.tensor([lens[i] - 1 for i in live], dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    outs = []
    for ready, pend in ((False, 0), (True, 0), (True, 1)):
        for _ in range(3):
            fc.append(kn[live], kn[live], sl, pos)
            out = fc.decode_attention(q, slots, cl, scale, out_dtype=torch.float32, num_ctas=9,
                                      tables_ready=ready, pending_tail=pend)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        outs.append(out.cpu())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    assert torch.all(outs[1][0] == 0)
    fc.close()


def test_flat_growth_release_and_bounds():
    dtype, Hq, Hk, D = torch.float16, 8, 2, 128
    fc, hk, hv = make_flat(dtype, 3, 20480, Hk, D, [100, 0, 0], seed=86)
    inf = fc.info()
    per_chunk = inf.granularity // (Hk * D * 2)
    # grow slot 0 past one chunk and write the new rows
    L2 = per_chunk + 50
    fc.reserve(0, L2)
    g = torch.Generator().manual_seed(87)
    k = torch.randn(L2 - 100, Hk, D, generator=g).to(dtype)
    v = torch.randn(L2 - 100, Hk, D, generator=g).to(dtype)
    hk[0, 100:L2], hv[0, 100:L2] = k, v
    fc.append(k.cuda(), v.cuda(), torch.zeros(L2 - 100, dtype=torch.int32, device="cuda"),
              torch.arange(100, L2, dtype=torch.int32, device="cuda"))
    q = torch.randn(1, Hq, D, generator=g).to(dtype)
    scale = 1.0 / math.sqrt(D)
    out = fc.decode_attention(q.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"),
                              torch.tensor([L2], dtype=torch.int32, device="cuda"), scale,
                              out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    want = oracle.decode_flat(q, hk, hv, torch.tensor([0], dtype=torch.int32),
                              torch.tensor([L2], dtype=torch.int32), scale)
    assert float(np.max(np.abs(out.double().cpu().numpy() - want))) <= 2e-3
    assert fc.info().committed_bytes == 2 * 2 * inf.granularity      # K and V, two chunks each
    # slot 1 holds nothing: a decode over it is clamped to zero tokens
    out = fc.decode_attention(q.cuda(), torch.ones(1, dtype=torch.int32, device="cuda"),
                              torch.tensor([10], dtype=torch.int32, device="cuda"), scale,
                              out_dtype=torch.float32)
    assert binding.get_error() == binding.DEVERR_CONTEXT
    assert torch.all(out == 0)
    # appends past the committed tokens, or to a bad slot, are refused
    kk = torch.randn(2, Hk, D, generator=g).to(dtype).cuda()
    fc.append(kk, kk, torch.tensor([2, 9], dtype=torch.int32, device="cuda"),
              torch.tensor([0, 0], dtype=torch.int32, device="cuda"))
    assert binding.get_error() == binding.DEVERR_SLOT
    # release slot 0: its memory is unmapped and its length clamps to zero
    fc.release(0)
    assert fc.info().committed_bytes == 0
    out = fc.decode_attention(q.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"),
                              torch.tensor([L2], dtype=torch.int32, device="cuda"), scale,
                              out_dtype=torch.float32)
    assert binding.get_error() == binding.DEVERR_CONTEXT and torch.all(out == 0)
    fc.close()
