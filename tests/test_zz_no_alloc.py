"""pkv_decode_attention_static: decode attention for callers that cannot
allocate device memory (a program whose device-memory budget all belongs to
its KV-cache pool, a plug-in limited to memory its host framework owns, code
where cudaMalloc's device synchronisation is not allowed). Instead of a
caller workspace it uses a fixed scratch array inside the library.

Checks, through the C ABI, that two calls in a row (different batches, so the
second finds the first's partials in the shared scratch and relies on the
first having put the split-K arrival counters back to zero) match the
ordinary workspace entry point within the decode tolerance, and that a shape
needing more scratch than the fixed array is refused. Kept in a file that
pytest collects last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

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


def _case(seed, lengths):
    spec = W.WorkloadSpec("no_alloc", len(lengths), 32, 8, 128, 16, "bf16", 1.0)
    st, v = W.make_workload(spec, seed=seed, lengths=lengths)
    dev = "cuda"
    kp, vp = v["k_pool"].to(dev), v["v_pool"].to(dev)
    binding.append(v["k_new"].to(dev), v["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    return v["q"].to(dev), kp, vp, st.block_tables.to(dev), st.context_lens.to(dev)


def test_static_scratch_matches_workspace_entry_point(L):
    scale = 1.0 / math.sqrt(128)
    cases = [_case(21, [1, 70, 513, 1500, 4096, 64, 2000, 333]),
             _case(22, [3000, 17, 900, 4000])]
    binding.get_error()
    for q, kp, vp, bt, cl in cases:          # two calls in a row, different batches
        ref = binding.decode_attention(q, kp, vp, bt, cl, scale, out_dtype=torch.float32)
        out = torch.full_like(ref, float("nan"))
        assert _static(L, q, kp, vp, bt, cl, scale, out) == 0, \
            L.pkv_last_error_message().decode()
        torch.cuda.synchronize()
        err = float((out.double() - ref.double()).abs().max())
        assert torch.isfinite(out).all() and err <= 2e-3, err
    assert binding.get_error() == 0


def test_static_scratch_refuses_shapes_that_do_not_fit(L):
    # q heads per kv head 16 at head_dim 128: one CTA per SM needs
    # 16 x 4096 + SMs x 8 x 16 x 132 bytes of scratch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = 16 * 4096 + sms * 8 * 16 * 132
    spec = W.WorkloadSpec("no_alloc_big", 2, 64, 4, 128, 16, "bf16", 1.0)
    st, v = W.make_workload(spec, seed=23, lengths=[100, 200])
    dev = "cuda"
    q, kp, vp = v["q"].to(dev), v["k_pool"].to(dev), v["v_pool"].to(dev)
    binding.append(v["k_new"].to(dev), v["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    rc = _static(L, q, kp, vp, st.block_tables.to(dev), st.context_lens.to(dev), 0.088, out)
    if need > STATIC_SCRATCH_BYTES:
        assert rc == -6 and b"fixed scratch" in L.pkv_last_error_message()
    else:
        assert rc == 0
