"""Byte accounting of bench.py (the numerator of every GB/s figure and of the
roofline fraction): the algorithmic bytes of one decode launch are the K and V
rows of every context token, q in and out, one table entry per used block and
one length per sequence; a block that several sequences share counts once in
the unique-bytes figure of the shared-prefix workload."""
import math

import bench
from paged_kv_cache_47_gb300 import workloads as W


def test_llama_decode_bytes():
    spec = W.SPECS[1]
    st = W.make_structure(spec, 0)
    lens = [int(x) for x in st.context_lens]
    assert sum(lens) == 155979
    row = bench.cache_row_bytes(spec, None)
    assert row == 128 * 2
    decode, append = bench.step_bytes(st, spec, row)
    kv = sum(lens) * 2 * 8 * 128 * 2
    qo = 64 * 32 * 128 * 2 * 2
    tables = sum(math.ceil(L / 16) for L in lens) * 4
    assert decode == kv + qo + tables + 4 * 64
    assert decode == 639977916          # the figure the ncu summary divides by
    # the append reads the new rows and writes them (plus the 8-byte slots)
    assert append == 64 * 8 * 2 * (128 * 2 + 128 * 2) + 8 * 64


def test_quantized_rows_carry_a_scale():
    spec = W.SPECS[1]
    assert bench.cache_row_bytes(spec, "int8") == 128 + 4
    assert bench.cache_row_bytes(spec, "fp8_e4m3") == 128 + 4


def test_shared_prefix_counts_once():
    spec = W.SPECS[3]
    st = W.make_structure(spec, 0)
    row = bench.cache_row_bytes(spec, None)
    lens = [int(x) for x in st.context_lens]
    uniq = bench.unique_kv_bytes(st, spec, row)
    # every sequence's rows once, minus the 19 repeats of the shared prefix
    # blocks; the step's tables are those after its copy-on-write, which gave
    # each sequence a private copy of the last of the 250 prefix blocks
    assert spec.cow and spec.shared_prefix % spec.block_size == 0
    shared_rows = spec.shared_prefix - spec.block_size
    want = (sum(lens) - (spec.num_seqs - 1) * shared_rows) * 2 * spec.num_kv_heads * row
    assert uniq == want
    assert uniq < sum(lens) * 2 * spec.num_kv_heads * row
