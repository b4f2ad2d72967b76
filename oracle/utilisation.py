"""KV-cache memory arithmetic — test infrastructure only.

The pages' memory model, written out as plain functions so the tests can pin
them to the numbers the pages print. Nothing here is on the GPU path.

- Per-token KV bytes: 2 x n_layers x n_kv_heads x head_dim x dtype_bytes
  ("PagedAttention — Math + Memory Model", section "The KV cache is big, and it
  grows").
- Contiguous utilisation U = L / L_max (same page, section "The fragmentation
  math").
- Paged utilisation U = L / (ceil(L/B) * B); waste per sequence at most B-1
  tokens, on average (B-1)/2 (same page, section "Why fragmentation nearly
  vanishes").
- Concurrency = floor(free KV memory / per-request footprint) (same page,
  section "A worked example").
"""
from __future__ import annotations

import math


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    return 2 * n_layers * n_kv_heads * head_dim * dtype_bytes


def u_contig(L: int, L_max: int) -> float:
    return L / L_max


def paged_slots(L: int, B: int) -> int:
    """Slots a sequence of L tokens holds under paging: ceil(L/B) blocks of B."""
    return math.ceil(L / B) * B


def u_paged(L: int, B: int) -> float:
    return L / paged_slots(L, B)


def paged_waste_tokens(L: int, B: int) -> int:
    return paged_slots(L, B) - L


def paged_worst_waste(B: int) -> int:
    return B - 1


def paged_mean_waste(B: int) -> float:
    """Mean unused slots in the last block, L mod B uniform over 0..B-1."""
    return sum(paged_waste_tokens(r if r else B, B) for r in range(B)) / B


def contiguous_request_bytes(L_max: int, bytes_per_token: float) -> float:
    return L_max * bytes_per_token


def paged_request_bytes(L: int, B: int, bytes_per_token: float) -> float:
    return paged_slots(L, B) * bytes_per_token


def concurrency(free_bytes: float, per_request_bytes: float) -> int:
    return int(math.floor(free_bytes / per_request_bytes + 1e-12))


def contiguous_waste_fraction(live_tokens_each: int, reserved_tokens_each: int) -> float:
    """Fraction of a contiguous reservation that holds no token."""
    return 1.0 - live_tokens_each / reserved_tokens_each
