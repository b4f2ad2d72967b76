"""End to end through the block manager: decode steps whose slots, copies and
block tables come from libpkv's C++ manager, with the K/V writes, copies and
attention on the GPU; the CPU side runs the block-manager oracle and the
decode oracle on its own copy of the pools.

Requests share a prompt prefix by hash, others have private prompts, one is
forked into beams (copy-on-write on their first divergent token), and one
is dropped half way. Slots and copies must equal the oracle's, pools must be
byte-exact, outputs within 2e-3.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from oracle.block_manager import BlockManagerOracle
from paged_kv_cache_47_gb300 import binding, build

pytestmark = pytest.mark.gpu

NB, B, HK, HQ, D = 256, 16, 2, 8, 128
DT = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


class Both:
    """The C++ manager and the oracle, driven with the same calls."""

    def __init__(self):
        self.bm = binding.BlockManager(NB, B)
        self.ref = BlockManagerOracle(NB, B)

    def add(self, seq, hashes=()):
        h = self.bm.add_sequence(seq, hashes)
        assert h == self.ref.add_sequence(seq, hashes)
        return h

    def append(self, seq, n):
        got = self.bm.append(seq, n)
        assert got == self.ref.append(seq, n)
        return got

    def fork(self, p, c):
        self.bm.fork(p, c)
        self.ref.fork(p, c)

    def free(self, s):
        self.bm.free_sequence(s)
        self.ref.free_sequence(s)


def test_decode_steps_driven_by_the_block_manager():
    g = torch.Generator().manual_seed(61)
    kp = torch.full((NB, HK, B, D), float("nan")).to(DT)
    vp = kp.clone()
    kg, vg = kp.cuda(), vp.cuda()
    m = Both()

    def write(slots):
        """Write fresh K/V rows at `slots` on both sides (append)."""
        n = len(slots)
        kn = torch.randn(n, HK, D, generator=g).to(DT)
        vn = torch.randn(n, HK, D, generator=g).to(DT)
        sl = torch.tensor(slots, dtype=torch.int64)
        oracle.append(kn, vn, sl, kp, vp)
        binding.append(kn.cuda(), vn.cuda(), sl.cuda(), kg, vg)

    def copy(pairs):
        if pairs:
            oracle.block_copy(pairs, kp, vp)
            binding.block_copy(pairs, kg, vg)

    # requests 0..2 share a 64-token system prompt (4 full blocks)
    prefix = [0x5eed0000 + i for i in range(4)]
    for s in range(3):
        hits = m.add(s, prefix)
        if not any(hits):               # the first request computes the prefix
            t = m.bm.table(s)
            write([b * B + o for b in t for o in range(B)])
        slots, pairs = m.append(s, 10 + 7 * s)    # the rest of each prompt
        copy(pairs)
        write(slots)
    # requests 3..5 have private prompts
    for s, L in zip(range(3, 6), (1, 33, 200)):
        m.add(s)
        slots, pairs = m.append(s, L)
        copy(pairs)
        write(slots)
    # request 1 forks into two beams that share its blocks
    m.fork(1, 6)
    m.fork(1, 7)
    live = [0, 1, 2, 3, 4, 5, 6, 7]
    scale = 1.0 / math.sqrt(D)
    for step in range(6):
        if step == 3:
            m.free(4)
            live.remove(4)
        slots, all_pairs = [], []
        for s in live:                   # one new token per live sequence
            sl, pairs = m.append(s, 1)
            slots += sl
            all_pairs += pairs
        copy(all_pairs)
        write(slots)
        tables, lens = m.bm.block_tables(live, 32)
        rt = torch.full((len(live), 32), -1, dtype=torch.int32)
        for i, s in enumerate(live):
            t = m.ref.table(s)
            rt[i, :len(t)] = torch.tensor(t, dtype=torch.int32)
        assert torch.equal(tables, rt)
        assert lens.tolist() == [m.ref.lens[s] for s in live]
        q = torch.randn(len(live), HQ, D, generator=g).to(DT)
        out = binding.decode_attention(q.cuda(), kg, vg, tables.cuda(), lens.cuda(), scale,
                                       out_dtype=torch.float32, num_ctas=7)
        torch.cuda.synchronize()
        assert binding.get_error() == 0
        want = oracle.decode(q, kp, vp, tables, lens, scale)
        err = float(np.max(np.abs(out.double().cpu().numpy() - want)))
        assert err <= 2e-3, (step, err)
    assert m.ref.ref == [m.bm.refcount(b) for b in range(NB)]
    assert torch.equal(kg.cpu().view(torch.int16), kp.view(torch.int16))
    assert torch.equal(vg.cpu().view(torch.int16), vp.view(torch.int16))
