"""Seeded synthetic decode workloads for the paged KV cache.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests. It draws shapes, context lengths, block tables, copy-on-write pairs,
append slots and tensor values. It holds none of the attention arithmetic.

Layout conventions (all tensors row-major, contiguous):
  q              [S][Hq][D]        dtype T
  k_pool, v_pool [NB][Hk][B][D]    dtype T   (one (block, kv head) chunk is B*D
                                              contiguous elements)
  block_tables   [S][M] int32, -1 past a sequence's last block
  context_lens   [S]    int32      length AFTER this step's append
  k_new, v_new   [S][Hk][D]        dtype T   (one new token per sequence)
  slot_mapping   [S]    int64      slot = physical_block * B + offset
  cow_pairs      [n][2] int64      (src, dst) physical block ids

Block tables map logical block i (tokens i*B .. i*B+B-1) to a physical block,
as in "PagedAttention — Math + Memory Model", section "PagedAttention: blocks
and the block table"; physical blocks are drawn from a random permutation of
the pool, so that neighbours in a sequence are scattered, as in the example
block table of "KV-cache paging in vLLM", section "PagedAttention: Paging for
KV-Caches".

Every pool position that no context may read (unused blocks, the tail of each
sequence's last block, the slot the append is about to fill) holds NaN, so a
kernel that reads past a context length or skips the append cannot pass a
parity test by accident.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
# dtype codes shared with the C ABI (pkv_dtype in include/pkv.h)
DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    std: float
    len_lo: int = 1
    len_hi: int = 1
    pool_ratio: float = 1.0          # NB = ceil(ratio * blocks needed)
    pool_blocks: Optional[int] = None  # fixed NB (overrides ratio)
    shared_prefix: int = 0           # tokens of a prefix shared by all sequences
    suffix_lo: int = 0
    suffix_hi: int = 0
    cow: bool = False                # copy-on-write of the last shared block

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def with_block_size(self, b: int) -> "WorkloadSpec":
        return replace(self, block_size=b)


# The five decode workloads. Index 1 is the headline (Llama-3-8B-shaped) case.
SPECS: List[WorkloadSpec] = [
    WorkloadSpec("tiny_fp32", 4, 4, 4, 64, 16, "f32", 1.0, 1, 100, pool_blocks=64),
    WorkloadSpec("llama3_8b_gqa4_bf16", 64, 32, 8, 128, 16, "bf16", 1.0, 512, 4096,
                 pool_ratio=1.2),
    WorkloadSpec("opt13b_mha_fp16", 256, 40, 40, 128, 16, "f16", 0.5, 128, 2048),
    WorkloadSpec("agent_swarm_prefix_fp16", 20, 32, 8, 128, 16, "f16", 1.0,
                 shared_prefix=4000, suffix_lo=0, suffix_hi=28000, cow=True),
    WorkloadSpec("long_ctx_70b_gqa8_bf16", 8, 64, 8, 128, 16, "bf16", 1.0, 32768, 131072),
]


@dataclass
class Structure:
    """Integer structure of one decode step (always on the CPU)."""
    spec: WorkloadSpec
    context_lens: torch.Tensor        # [S] int32
    block_tables: torch.Tensor        # [S][M] int32 (after copy-on-write)
    block_tables_pre_cow: torch.Tensor  # [S][M] int32 (before copy-on-write)
    num_blocks: int
    slot_mapping: torch.Tensor        # [S] int64
    cow_pairs: torch.Tensor           # [n][2] int64
    nan_positions: List[tuple] = field(default_factory=list)  # (block, first_off, last_off_excl)
    used_blocks: Optional[torch.Tensor] = None  # bool [NB], referenced before CoW

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max().item()) if self.context_lens.numel() else 0


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def make_structure(spec: WorkloadSpec, seed: int = 0,
                   lengths: Optional[List[int]] = None) -> Structure:
    """Draw context lengths, the physical block permutation and the tables.

    Draw order on one CPU generator seeded with `seed`: lengths, then the
    permutation of physical blocks. `lengths` overrides the drawn lengths
    (used by edge-case tests).
    """
    g = torch.Generator().manual_seed(seed)
    S, B = spec.num_seqs, spec.block_size
    P = spec.shared_prefix
    if lengths is not None:
        lens = torch.tensor(lengths, dtype=torch.int64)
        S = lens.numel()
    elif P > 0:
        suffix = torch.randint(spec.suffix_lo, spec.suffix_hi + 1, (S,), generator=g)
        lens = P + suffix
    else:
        lens = torch.randint(spec.len_lo, spec.len_hi + 1, (S,), generator=g)
    lens_l = [int(x) for x in lens.tolist()]

    if P > 0:
        n_prefix = _cdiv(P, B)
        priv_counts = [max(0, _cdiv(L, B) - n_prefix) for L in lens_l]
        spare = (S - 1) if spec.cow else 0
        need = n_prefix + sum(priv_counts) + spare
    else:
        n_prefix = 0
        priv_counts = [_cdiv(L, B) for L in lens_l]
        spare = 0
        need = sum(priv_counts)
    if spec.pool_blocks is not None:
        NB = max(spec.pool_blocks, need)
    else:
        NB = max(1, math.ceil(spec.pool_ratio * need))
    perm = torch.randperm(NB, generator=g).tolist()

    M = max(1, max((_cdiv(L, B) for L in lens_l), default=1))
    tables = torch.full((S, M), -1, dtype=torch.int32)
    cursor = 0
    prefix_ids = perm[cursor:cursor + n_prefix]
    cursor += n_prefix
    for s, L in enumerate(lens_l):
        nblk = _cdiv(L, B)
        row = list(prefix_ids[:min(n_prefix, nblk)])
        k = nblk - len(row)
        row += perm[cursor:cursor + k]
        cursor += k
        if row:
            tables[s, :len(row)] = torch.tensor(row, dtype=torch.int32)
    spares = perm[cursor:cursor + spare]
    cursor += spare

    used = torch.zeros(NB, dtype=torch.bool)
    for s, L in enumerate(lens_l):
        nblk = _cdiv(L, B)
        if nblk:
            used[tables[s, :nblk].long()] = True

    pre_cow = tables.clone()
    pairs = []
    if spec.cow and n_prefix > 0 and S > 1:
        # Copy-on-write of the last shared block: a writer that still shares the
        # block with others copies it to a fresh block, repoints its table entry
        # and drops one reference; the last holder keeps the original
        # ("PagedAttention — Math + Memory Model", section "Copy-on-write").
        last = n_prefix - 1
        shared = int(pre_cow[0, last])
        refcount = sum(1 for L in lens_l if _cdiv(L, B) > last)
        spare_it = iter(spares)
        for s, L in enumerate(lens_l):
            if _cdiv(L, B) <= last or refcount <= 1:
                continue
            fresh = next(spare_it)
            pairs.append((shared, fresh))
            tables[s, last] = fresh
            refcount -= 1

    # slot of the token this step appends: position L-1 of each sequence
    slots = torch.full((S,), -1, dtype=torch.int64)
    for s, L in enumerate(lens_l):
        if L > 0:
            p = L - 1
            slots[s] = int(tables[s, p // B]) * B + p % B

    # NaN sentinels: tails of last blocks and the pre-append slot (only where
    # the block is private before copy-on-write, so shared data stays valid)
    refc = {}
    for s, L in enumerate(lens_l):
        for j in range(_cdiv(L, B)):
            b = int(pre_cow[s, j])
            refc[b] = refc.get(b, 0) + 1
    nan_pos = []
    for s, L in enumerate(lens_l):
        if L == 0:
            continue
        last_blk = int(pre_cow[s, (L - 1) // B])
        if refc[last_blk] == 1:
            nan_pos.append((last_blk, (L - 1) % B, B))
        elif L % B:
            nan_pos.append((last_blk, L % B, B))

    return Structure(spec=spec, context_lens=lens.to(torch.int32), block_tables=tables,
                     block_tables_pre_cow=pre_cow, num_blocks=NB, slot_mapping=slots,
                     cow_pairs=torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2),
                     nan_positions=nan_pos, used_blocks=used)


_CHUNK = 1 << 24  # elements drawn per generator call (fixes the draw sequence)


def _randn(shape, std, dtype, gen, device):
    n = 1
    for x in shape:
        n *= x
    out = torch.empty(n, dtype=dtype, device=device)
    for i in range(0, n, _CHUNK):
        m = min(_CHUNK, n - i)
        out[i:i + m] = (torch.randn(m, generator=gen, device=device) * std).to(dtype)
    return out.view(*shape)


def make_values(st: Structure, seed: int = 0, device="cpu") -> dict:
    """Draw q, the K/V pools and the new token's K/V on `device`.

    Values are N(0, std^2) drawn in fp32 and rounded to the workload dtype, so
    every consumer sees the same dtype-rounded numbers. Draw order on one
    generator (seeded with seed+1) on `device`: q, K pool, V pool, k_new, v_new.
    """
    sp = st.spec
    dt = DTYPES[sp.dtype]
    S = st.context_lens.numel()
    gen = torch.Generator(device=device).manual_seed(seed + 1)
    q = _randn((S, sp.num_q_heads, sp.head_dim), sp.std, dt, gen, device)
    shape = (st.num_blocks, sp.num_kv_heads, sp.block_size, sp.head_dim)
    k_pool = _randn(shape, sp.std, dt, gen, device)
    v_pool = _randn(shape, sp.std, dt, gen, device)
    k_new = _randn((S, sp.num_kv_heads, sp.head_dim), sp.std, dt, gen, device)
    v_new = _randn((S, sp.num_kv_heads, sp.head_dim), sp.std, dt, gen, device)
    nan = float("nan")
    unused = (~st.used_blocks).nonzero().flatten()
    if unused.numel():
        idx = unused.to(device)
        k_pool[idx] = nan
        v_pool[idx] = nan
    for (b, lo, hi) in st.nan_positions:
        k_pool[b, :, lo:hi, :] = nan
        v_pool[b, :, lo:hi, :] = nan
    return dict(q=q, k_pool=k_pool, v_pool=v_pool, k_new=k_new, v_new=v_new)


def make_workload(index_or_spec, seed: int = 0, device="cpu", block_size: Optional[int] = None,
                  lengths: Optional[List[int]] = None, **overrides):
    """Structure + values for one of SPECS (or a custom spec)."""
    spec = SPECS[index_or_spec] if isinstance(index_or_spec, int) else index_or_spec
    if block_size is not None:
        spec = spec.with_block_size(block_size)
    if overrides:
        spec = replace(spec, **overrides)
    st = make_structure(spec, seed, lengths=lengths)
    vals = make_values(st, seed, device)
    return st, vals
