"""The C++ block manager (pkv_bm_* in libpkv) against the block-manager oracle.

Bookkeeping is integer work, so parity is exact: on random operation
sequences every call's slots, copies and failures, and after every call all
tables, reference counts and free counts, must equal the oracle's. The
utilisation simulator must reproduce the pages' worked examples.
"""
import json
import math
import os
import random

import pytest

from oracle import utilisation as U
from oracle.block_manager import BlockManagerOracle, OutOfBlocks
from paged_kv_cache_47_gb300 import binding, build

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "utilisation.json")))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


def _same_state(bm, ref, live):
    for s in live:
        assert bm.table(s) == ref.table(s), s
    assert [bm.refcount(b) for b in range(ref.num_blocks)] == ref.ref
    st = bm.stats()
    assert st.free_blocks == ref.num_free()
    assert st.tokens == ref.tokens() and st.sequences == len(ref.tables)
    assert st.prefix_entries == len(ref.by_hash)


@pytest.mark.parametrize("seed,NB,B", [(1, 48, 8), (2, 64, 16), (3, 20, 4), (4, 200, 16)])
def test_random_operations_match_the_oracle(seed, NB, B):
    rng = random.Random(seed)
    bm, ref = binding.BlockManager(NB, B), BlockManagerOracle(NB, B)
    live, next_id = [], 0
    for step in range(2500):
        op = rng.random()
        if op < 0.2 or not live:
            chain = [rng.randrange(4) for _ in range(rng.randrange(4))]
            hashes = [(hash(tuple(chain[:i + 1])) * 2654435761) % (2 ** 64)
                      for i in range(len(chain))]
            try:
                want = ref.add_sequence(next_id, hashes)
            except OutOfBlocks:
                with pytest.raises(binding.NoBlocks):
                    bm.add_sequence(next_id, hashes)
            else:
                assert bm.add_sequence(next_id, hashes) == want
                live.append(next_id)
                next_id += 1
        elif op < 0.6:
            s, n = rng.choice(live), rng.randrange(0, 3 * B)
            try:
                want = ref.append(s, n)
            except OutOfBlocks:
                with pytest.raises(binding.NoBlocks):
                    bm.append(s, n)
            else:
                assert bm.append(s, n) == want, (step, s, n)
        elif op < 0.75:
            p = rng.choice(live)
            ref.fork(p, next_id)
            bm.fork(p, next_id)
            live.append(next_id)
            next_id += 1
        else:
            s = rng.choice(live)
            ref.free_sequence(s)
            bm.free_sequence(s)
            live.remove(s)
        _same_state(bm, ref, live)


def test_block_tables_for_decode():
    bm = binding.BlockManager(16, 16)
    for s, L in enumerate([40, 1, 16]):
        bm.add_sequence(s)
        bm.append(s, L)
    tables, lens = bm.block_tables([2, 0, 1], 4)
    assert lens.tolist() == [16, 40, 1]
    assert tables.tolist() == [[4, -1, -1, -1], [0, 1, 2, -1], [3, -1, -1, -1]]
    with pytest.raises(binding.PkvError):
        bm.block_tables([0], 2)            # three blocks do not fit two columns
    with pytest.raises(binding.PkvError):
        bm.block_tables([7], 4)            # unknown sequence


def test_errors_change_nothing():
    bm = binding.BlockManager(4, 16)
    bm.add_sequence(0)
    bm.append(0, 20)
    with pytest.raises(binding.PkvError):
        bm.add_sequence(0)                 # exists
    with pytest.raises(binding.PkvError):
        bm.fork(0, 0)                      # child exists
    with pytest.raises(binding.PkvError):
        bm.fork(9, 1)                      # unknown parent
    with pytest.raises(binding.PkvError):
        bm.free_sequence(9)
    with pytest.raises(binding.NoBlocks):
        bm.append(0, 60)                   # 80 tokens need 5 blocks
    assert bm.table(0) == [0, 1] and bm.num_free() == 2
    bm.fork(0, 1)
    # a copy is needed but the caller gave no room for it
    L = binding._bm_lib()
    import ctypes
    slots = (ctypes.c_int64 * 1)()
    nc = ctypes.c_int32(0)
    assert L.pkv_bm_append(bm._h, 1, 1, slots, None, 0, ctypes.byref(nc)) == -1
    assert bm.table(1) == [0, 1] and bm.refcount(1) == 2


def test_simulator_reproduces_the_worked_example():
    w = GOLDEN["worked_example"]
    budget_kib = w["free_gb"] * 1024 * 1024
    B, L, L_max = w["B"], w["L"], w["L_max"]
    blocks = budget_kib // (B * w["kb_per_token"])
    adm, u = binding.simulate_admission(blocks, B, [L] * 200)
    assert adm == w["paged_requests"] and u == pytest.approx(U.u_paged(L, B))
    adm, u = binding.simulate_admission(blocks, B, [L] * 200, reserve_tokens=L_max)
    assert adm == w["contiguous_requests"]
    assert u == pytest.approx(U.u_contig(L, L_max))


def test_simulator_reproduces_the_rdna4_budget():
    r = GOLDEN["rdna4_swarm"]
    mbpt = r["mb_per_token"]
    budget_mb = r["kv_budget_gb"] * 1000
    B = r["paged_16"]["B"]
    blocks = int(budget_mb // (B * mbpt))
    live = r["reserve_8k"]["live_tokens_each"]
    # reserve-for-max at 16k (in block units) admits 4 of 8 agents
    adm, _ = binding.simulate_admission(blocks, B, [live] * r["agents"],
                                        reserve_tokens=r["reserve_16k"]["tokens"])
    assert adm == r["reserve_16k"]["admitted"]
    # at 8k all 8 fit, and most of what they hold is empty
    adm, u = binding.simulate_admission(blocks, B, [live] * r["agents"],
                                        reserve_tokens=r["reserve_8k"]["tokens"])
    assert adm == r["reserve_8k"]["admitted"]
    # 1 - 3000/8000 = 62.5 %, which the page prints rounded half up
    assert math.floor(100 * (1 - u) + 0.5) == r["reserve_8k"]["wasted_percent"]
    # paged: all 8 fit with under 1 % waste
    adm, u = binding.simulate_admission(blocks, B, [live] * r["agents"])
    assert adm == r["agents"] and 100 * (1 - u) < r["paged_16"]["wasted_below_percent"]


def test_simulator_utilisation_on_mixed_lengths():
    rng = random.Random(5)
    lens = [rng.randrange(1, 3000) for _ in range(300)]
    adm, u = binding.simulate_admission(100000, 16, lens)
    assert adm == 300
    assert u == pytest.approx(sum(lens) / sum(U.paged_slots(L, 16) for L in lens))
    adm, _ = binding.simulate_admission(1000, 16, lens)
    used = 0
    for i, L in enumerate(lens):       # admission stops at the first request that does not fit
        if used + math.ceil(L / 16) > 1000:
            assert adm == i
            break
        used += math.ceil(L / 16)


def test_append_batch_equals_appends_in_order():
    rng = random.Random(11)
    bm, ref = binding.BlockManager(60, 8), BlockManagerOracle(60, 8)
    for s in range(6):
        bm.add_sequence(s)
        ref.add_sequence(s)
    bm.fork(2, 6)
    ref.fork(2, 6)
    ids = list(range(7))
    for step in range(40):
        counts = [rng.randrange(0, 6) for _ in ids]
        want_slots, want_pairs, failed = [], [], None
        for i, (s, n) in enumerate(zip(ids, counts)):
            try:
                sl, pr = ref.append(s, n)
            except OutOfBlocks:
                failed = i
                break
            want_slots += sl
            want_pairs += pr
        if failed is None:
            slots, pairs = bm.append_batch(ids, counts)
            assert slots.tolist() == want_slots
            assert [tuple(p) for p in pairs.tolist()] == want_pairs
        else:
            with pytest.raises(binding.NoBlocks):
                bm.append_batch(ids, counts)
        _same_state(bm, ref, ids)
        if failed is not None:
            break
    assert failed is not None          # the pool ran out on the way


def test_prepared_step_equals_list_calls():
    # two managers fed the same operations: one through the list-taking calls,
    # one through a prepared step (buffers made once); the forked sequence
    # makes its first append copy a shared block
    a, b = binding.BlockManager(80, 8), binding.BlockManager(80, 8)
    for bm in (a, b):
        for s in range(5):
            bm.add_sequence(s)
            bm.append(s, 2 + 5 * s)       # sequence 1: 7 tokens, a partial block
        bm.fork(1, 5)
    ids, counts = [0, 1, 2, 3, 4, 5], [1, 1, 2, 0, 1, 1]
    M = 16
    prep = b.prepared_step(ids, counts, M)
    for step in range(6):
        ws, wp = a.append_batch(ids, counts)
        gs, gp = prep.append()
        assert gs.tolist() == ws.tolist()
        assert gp.tolist() == wp.tolist()
        if step == 0:
            # sequences 1 and 5 share a partial last block: the first writer copies it
            assert len(wp) == 1
        wt, wl = a.block_tables(ids, M)
        gt, gl = prep.block_tables()
        assert gt.tolist() == wt.tolist() and gl.tolist() == wl.tolist()
    assert [a.table(s) for s in ids] == [b.table(s) for s in ids]
