"""pkv_decode_attention_static: decode attention for callers that cannot
allocate device memory (a program whose device-memory budget all belongs to
its KV-cache pool, a plug-in limited to memory its host framework owns, code
where cudaMalloc's device synchronisation is not allowed). Instead of a
caller workspace it uses a fixed scratch array inside the library.

Checks, through the C ABI, that calls in a row (different batches, so each
finds the previous call's partials in the shared scratch and relies on it
having put the split-K arrival counters back to zero) match both the ordinary
workspace entry point and the fp64 oracle within the decode tolerance, also
across head groupings (GQA 4, MHA, GQA 8) and for a batch longer than one
launch carries; and that a shape needing more scratch than the fixed array is
refused. Kept in a file that pytest collects last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_cache_47_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 2 << 20      # PKV_STATIC_SCRATCH_BYTES in include/pkv.h


@pytest.fixture(scope="module")
def L():
    build.build()
    lib = binding.lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.pkv_decode_attention_static.argtypes = [ctypes.POINTER(binding.CacheDesc), vp, i32, i32,
                                                vp, vp, vp, i32, vp, ctypes.c_float, vp, i32, vp]
    lib.pkv_decode_attention_static.restype = i32
    return lib


def _static(L, q, kp, vp, bt, cl, scale, out):
    desc = binding.cache_desc(kp)
    return L.pkv_decode_attention_static(
        ctypes.byref(desc), q.data_ptr(), q.shape[0], q.shape[1], kp.data_ptr(), vp.data_ptr(),
        bt.data_ptr(), bt.shape[1], cl.data_ptr(), scale, out.data_ptr(),
        binding.DTYPE_CODE[out.dtype], torch.cuda.current_stream().cuda_stream)


def _case(seed, lengths, hq=32, hk=8, d=128, dtype="bf16"):
    spec = W.WorkloadSpec("no_alloc", len(lengths), hq, hk, d, 16, dtype, 1.0)
    st, v = W.make_workload(spec, seed=seed, lengths=lengths)
    dev = "cuda"
    kp, vp = v["k_pool"].to(dev), v["v_pool"].to(dev)
    binding.append(v["k_new"].to(dev), v["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    # the oracle's own copy of the post-append cache
    kp_o, vp_o = v["k_pool"].clone(), v["v_pool"].clone()
    oracle.append(v["k_new"], v["v_new"], st.slot_mapping, kp_o, vp_o)
    ref = oracle.decode(v["q"], kp_o, vp_o, st.block_tables, st.context_lens,
                        1.0 / math.sqrt(d))
    return (v["q"].to(dev), kp, vp, st.block_tables.to(dev), st.context_lens.to(dev)), ref


def _check_calls(L, cases):
    binding.get_error()
    for (q, kp, vp, bt, cl), ref in cases:       # calls in a row on the shared scratch
        scale = 1.0 / math.sqrt(q.shape[2])
        ws_out = binding.decode_attention(q, kp, vp, bt, cl, scale, out_dtype=torch.float32)
        out = torch.full_like(ws_out, float("nan"))
        assert _static(L, q, kp, vp, bt, cl, scale, out) == 0, \
            L.pkv_last_error_message().decode()
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        err_ws = float((out.double() - ws_out.double()).abs().max())
        err_oracle = float(np.abs(out.double().cpu().numpy() - ref).max())
        assert err_ws <= 2e-3 and err_oracle <= 2e-3, (err_ws, err_oracle)
    assert binding.get_error() == 0


def test_static_scratch_matches_workspace_entry_point(L):
    _check_calls(L, [_case(21, [1, 70, 513, 1500, 4096, 64, 2000, 333]),
                     _case(22, [3000, 17, 900, 4000])])


def test_static_scratch_across_head_groupings(L):
    # the partials' layout in the scratch changes with the q heads per kv
    # head: GQA 4, then MHA, then GQA 8, then GQA 4 again
    _check_calls(L, [_case(24, [700, 65, 2049], 32, 8),
                     _case(25, [129, 1000, 1, 64, 3000], 40, 40, 128, "f16"),
                     _case(26, [5000, 33], 64, 8),
                     _case(27, [4096, 512], 32, 8)])


def test_static_scratch_batch_longer_than_one_launch(L):
    # 1100 sequences: the library launches the batch in two pieces that use
    # the same scratch one after the other
    g = torch.Generator().manual_seed(28)
    lengths = torch.randint(1, 41, (1100,), generator=g).tolist()
    _check_calls(L, [_case(28, lengths, 8, 8, 64, "f16"), _case(29, [300, 2], 8, 8, 64, "f16")])


def test_static_scratch_refuses_shapes_that_do_not_fit(L):
    # q heads per kv head 16 at head_dim 128: one CTA per SM needs
    # 16 x 4096 + SMs x 8 x 16 x 132 bytes of scratch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = 16 * 4096 + sms * 8 * 16 * 132
    if need <= STATIC_SCRATCH_BYTES:
        pytest.skip(f"{sms} SMs: the 16-heads-per-kv-head shape fits the fixed scratch")
    spec = W.WorkloadSpec("no_alloc_big", 2, 64, 4, 128, 16, "bf16", 1.0)
    st, v = W.make_workload(spec, seed=23, lengths=[100, 200])
    dev = "cuda"
    q, kp, vp = v["q"].to(dev), v["k_pool"].to(dev), v["v_pool"].to(dev)
    binding.append(v["k_new"].to(dev), v["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    rc = _static(L, q, kp, vp, st.block_tables.to(dev), st.context_lens.to(dev), 0.088, out)
    assert rc == -6 and b"fixed scratch" in L.pkv_last_error_message()
