"""Pins of the block-manager oracle against the pages and closed forms.

- On-demand allocation and the paged waste bound ("PagedAttention — Math +
  Memory Model", sections "PagedAttention: blocks and the block table" and
  "Why fragmentation nearly vanishes"), cross-checked with the utilisation
  closed forms.
- Copy-on-write copies exactly the written block; the last holder writes in
  place; freeing returns a block at count zero (same page, section
  "Copy-on-write: sharing blocks across samples").
- Prefix sharing of a 4000-token prompt by 20 requests ("KV-Cache Optimization
  & PagedAttention for Long-Context Agents", "Key KV-Cache Optimization
  Principles", item 3).
- Admission counts found by allocating until the pool is full reproduce the
  pages' worked examples (tests/golden/utilisation.json).
- Invariants under random operation sequences.
"""
import json
import math
import os
import random

import pytest

from oracle import utilisation as U
from oracle.block_manager import BlockManagerOracle, OutOfBlocks

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "utilisation.json")))


def test_on_demand_allocation_and_waste_bound():
    B = 16
    for L in (1, 15, 16, 17, 255, 256, 257, 512, 3000):
        m = BlockManagerOracle(400, B)
        m.add_sequence(0)
        slots, copies = m.append(0, L)
        assert copies == []
        assert len(m.table(0)) == math.ceil(L / B) == m.used_blocks()
        assert m.table(0) == list(range(math.ceil(L / B)))      # a fresh pool hands out 0, 1, 2, ...
        assert slots == [m.table(0)[t // B] * B + t % B for t in range(L)]
        waste = m.used_blocks() * B - m.tokens()
        assert waste == U.paged_waste_tokens(L, B) <= U.paged_worst_waste(B)


def test_copy_on_write_copies_only_the_written_block():
    B = 16
    m = BlockManagerOracle(10, B)
    m.add_sequence(0)
    m.append(0, 20)                       # blocks 0 (full) and 1 (4 tokens)
    m.fork(0, 1)
    assert m.ref[0] == 2 and m.ref[1] == 2
    slots, copies = m.append(1, 1)        # the child writes into the shared block 1
    assert copies == [(1, 2)] and slots == [2 * B + 4]
    assert m.table(1) == [0, 2] and m.table(0) == [0, 1]
    assert m.ref[0] == 2 and m.ref[1] == 1 and m.ref[2] == 1
    slots, copies = m.append(0, 1)        # the last holder writes in place
    assert copies == [] and slots == [1 * B + 4]


def test_fork_at_a_block_boundary_needs_no_copy():
    m = BlockManagerOracle(10, 16)
    m.add_sequence(0)
    m.append(0, 32)
    m.fork(0, 1)
    slots, copies = m.append(1, 1)
    assert copies == [] and m.table(1) == [0, 1, 2] and slots == [2 * 16]


def test_blocks_return_to_the_pool_at_count_zero():
    m = BlockManagerOracle(8, 16)
    m.add_sequence(0)
    m.append(0, 40)
    m.fork(0, 1)
    m.fork(0, 2)
    assert m.num_free() == 5
    m.free_sequence(1)
    m.free_sequence(0)
    assert m.num_free() == 5              # sequence 2 still holds all three
    m.free_sequence(2)
    assert m.num_free() == 8 and all(r == 0 for r in m.ref)
    # the most recently freed block is taken first
    m.add_sequence(3)
    m.append(3, 1)
    assert m.table(3) == [2]


def test_shared_prompt_prefix_of_twenty_requests():
    B, prefix = 16, 4000
    n = prefix // B                       # 250 full blocks
    hashes = [1000 + i for i in range(n)]
    m = BlockManagerOracle(400, B)
    hits = [m.add_sequence(s, hashes) for s in range(20)]
    assert not any(hits[0]) and all(all(h) for h in hits[1:])
    assert m.used_blocks() == n and all(m.ref[b] == 20 for b in range(n))
    # each request continues privately after the shared prefix
    for s in range(20):
        _, copies = m.append(s, 1)
        assert copies == []               # the prefix ends on a block boundary
    assert m.used_blocks() == n + 20
    for s in range(20):
        m.free_sequence(s)
    assert m.num_free() == 400 and m.by_hash == {}


def test_out_of_blocks_changes_nothing():
    m = BlockManagerOracle(3, 16)
    m.add_sequence(0)
    m.append(0, 40)
    before = (m.table(0), m.num_free(), list(m.ref), m.lens[0])
    with pytest.raises(OutOfBlocks):
        m.append(0, 10)                   # 40 + 10 tokens need a fourth block
    assert (m.table(0), m.num_free(), list(m.ref), m.lens[0]) == before
    m.fork(0, 1)
    with pytest.raises(OutOfBlocks):
        m.append(1, 1)                    # the copy needs a free block
    assert m.table(1) == m.table(0)


def _admitted(num_blocks, B, L):
    """Requests of L tokens admitted by allocating until the pool is full."""
    m = BlockManagerOracle(num_blocks, B)
    n = 0
    while True:
        m.add_sequence(n)
        try:
            m.append(n, L)
        except OutOfBlocks:
            return n
        n += 1


def test_admission_by_allocation_reproduces_the_worked_example():
    w = GOLDEN["worked_example"]
    kib_per_token = w["kb_per_token"]
    budget_kib = w["free_gb"] * 1024 * 1024
    B = w["B"]
    blocks = budget_kib // (B * kib_per_token)
    assert _admitted(blocks, B, w["L"]) == w["paged_requests"]
    # reserve-for-max: one slab of L_max tokens per request
    assert budget_kib // (w["L_max"] * kib_per_token) == w["contiguous_requests"]


def test_admission_by_allocation_reproduces_the_rdna4_budget():
    r = GOLDEN["rdna4_swarm"]
    mb_per_token, budget_mb = r["mb_per_token"], r["kv_budget_gb"] * 1000
    assert int(budget_mb // (r["reserve_16k"]["tokens"] * mb_per_token)) == \
        r["reserve_16k"]["admitted"]
    # paged: 8 agents at 3000 live tokens each fit, and the whole budget
    # holds about 71k tokens in 16-token blocks
    B = r["paged_16"]["B"]
    blocks = int(budget_mb // (B * mb_per_token))
    m = BlockManagerOracle(blocks, B)
    for s in range(r["agents"]):
        m.add_sequence(s)
        m.append(s, r["reserve_8k"]["live_tokens_each"])
    waste = 100 * (m.used_blocks() * B - m.tokens()) / (m.used_blocks() * B)
    assert waste < r["paged_16"]["wasted_below_percent"]
    assert round(blocks * B / 1000) == r["paged_16"]["approx_aggregate_ktokens"]


def _check_invariants(m):
    count = [0] * m.num_blocks
    for t in m.tables.values():
        for b in t:
            count[b] += 1
    assert count == m.ref
    assert sorted(m.free) == [b for b in range(m.num_blocks) if m.ref[b] == 0]
    assert len(set(m.free)) == len(m.free)
    for s, t in m.tables.items():
        assert len(t) == math.ceil(m.lens[s] / m.B)
    for h, b in m.by_hash.items():
        assert m.hash_of[b] == h and m.ref[b] > 0


def test_invariants_under_random_operations():
    rng = random.Random(7)
    m = BlockManagerOracle(64, 8)
    live, next_id = [], 0
    for _ in range(3000):
        op = rng.random()
        try:
            if op < 0.25 or not live:
                hashes = [rng.randrange(6) for _ in range(rng.randrange(3))]
                # a prefix is a chain: a block's hash stands for everything before it
                hashes = [hash(tuple(hashes[:i + 1])) & 0xFFFFFFFF for i in range(len(hashes))]
                m.add_sequence(next_id, hashes)
                live.append(next_id)
                next_id += 1
            elif op < 0.6:
                m.append(rng.choice(live), rng.randrange(1, 20))
            elif op < 0.75:
                m.fork(rng.choice(live), next_id)
                live.append(next_id)
                next_id += 1
            else:
                s = rng.choice(live)
                m.free_sequence(s)
                live.remove(s)
        except OutOfBlocks:
            pass
        _check_invariants(m)
