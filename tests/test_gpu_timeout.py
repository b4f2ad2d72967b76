"""The bounded-wait failure path, made to run out on purpose without a fault.

Every wait on an on-chip barrier in the decode kernel gives up after a limit,
flags PKV_DEVERR_TIMEOUT in the device error word and ends its warp's work, so
the kernel returns instead of hanging. The library's test hook shortens the
limit and makes one launch's first CTA withhold one producer arrival (a
barrier phase that nothing completes). Checked here:
  - the call returns, and pkv_get_error reports PKV_ERR_TIMEOUT with the
    PKV_DEVERR_TIMEOUT bit;
  - the context stays usable: after the workspace is zeroed again (the
    documented recovery for a caller-owned workspace), the next call matches
    the oracle; for pkv_decode_attention_static, whose scratch pkv_get_error
    zeroes itself, the next call matches with no action by the caller;
  - with the short limit but no withheld arrival, calls complete normally.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from oracle import oracle
from paged_kv_cache_47_gb300 import binding, build, workloads as W

pytestmark = pytest.mark.gpu

PKV_ERR_TIMEOUT = -5
SHORT_NS = 2_000_000      # 2 ms: far above a healthy wait, far below the default 2 s


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()
    yield
    binding.set_wait_fault(0, 0)


@pytest.fixture
def case():
    spec = W.WorkloadSpec("timeout", 12, 32, 8, 128, 16, "bf16", 1.0)
    lengths = [700, 65, 2049, 1, 300, 4096, 1500, 17, 999, 3000, 128, 2500]
    st, v = W.make_workload(spec, seed=41, lengths=lengths)
    dev = "cuda"
    kp, vp = v["k_pool"].to(dev), v["v_pool"].to(dev)
    binding.append(v["k_new"].to(dev), v["v_new"].to(dev), st.slot_mapping.to(dev), kp, vp)
    kp_o, vp_o = v["k_pool"].clone(), v["v_pool"].clone()
    oracle.append(v["k_new"], v["v_new"], st.slot_mapping, kp_o, vp_o)
    ref = oracle.decode(v["q"], kp_o, vp_o, st.block_tables, st.context_lens, 1.0 / math.sqrt(128))
    torch.cuda.synchronize()
    binding.get_error()
    return (v["q"].to(dev), kp, vp, st.block_tables.to(dev), st.context_lens.to(dev)), ref


def _err(out, ref):
    return float(np.abs(out.double().cpu().numpy() - ref).max())


def test_short_limit_alone_changes_nothing(case):
    (q, kp, vp, bt, cl), ref = case
    binding.set_wait_fault(SHORT_NS, 0)
    try:
        for C in (0, 7):
            out = binding.decode_attention(q, kp, vp, bt, cl, 1.0 / math.sqrt(128),
                                           out_dtype=torch.float32, num_ctas=C)
            assert binding.get_error_status() == (0, 0)
            assert _err(out, ref) <= 2e-3
    finally:
        binding.set_wait_fault(0, 0)


def test_timed_out_wait_reports_and_workspace_recovers(case):
    (q, kp, vp, bt, cl), ref = case
    scale = 1.0 / math.sqrt(128)
    ws = binding.alloc_workspace(kp, 32)
    binding.set_wait_fault(SHORT_NS, 1)
    try:
        binding.decode_attention(q, kp, vp, bt, cl, scale, out_dtype=torch.float32, workspace=ws)
        status, word = binding.get_error_status()
    finally:
        binding.set_wait_fault(0, 0)
    assert status == PKV_ERR_TIMEOUT and word & binding.DEVERR_TIMEOUT
    ws.zero_()                               # the caller's recovery step
    out = binding.decode_attention(q, kp, vp, bt, cl, scale, out_dtype=torch.float32,
                                   workspace=ws)
    assert binding.get_error_status() == (0, 0)
    assert _err(out, ref) <= 2e-3
    counters = ws[: 4096 * 16].view(torch.int32)
    assert int(counters.abs().sum()) == 0


def test_timed_out_wait_static_scratch_recovers(case):
    (q, kp, vp, bt, cl), ref = case
    L = binding.lib()
    vp_, i32 = ctypes.c_void_p, ctypes.c_int32
    L.pkv_decode_attention_static.argtypes = [ctypes.POINTER(binding.CacheDesc), vp_, i32, i32,
                                              vp_, vp_, vp_, i32, vp_, ctypes.c_float, vp_, i32,
                                              vp_]
    L.pkv_decode_attention_static.restype = i32
    desc = binding.cache_desc(kp)
    scale = 1.0 / math.sqrt(128)

    def static(out):
        return L.pkv_decode_attention_static(
            ctypes.byref(desc), q.data_ptr(), q.shape[0], q.shape[1], kp.data_ptr(),
            vp.data_ptr(), bt.data_ptr(), bt.shape[1], cl.data_ptr(), scale, out.data_ptr(),
            binding.DTYPE_CODE[out.dtype], torch.cuda.current_stream().cuda_stream)

    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    binding.set_wait_fault(SHORT_NS, 1)
    try:
        assert static(out) == 0
        status, word = binding.get_error_status()    # also zeroes the static scratch
    finally:
        binding.set_wait_fault(0, 0)
    assert status == PKV_ERR_TIMEOUT and word & binding.DEVERR_TIMEOUT
    for _ in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        assert static(out) == 0
        assert binding.get_error_status() == (0, 0)
        assert _err(out, ref) <= 2e-3


def test_hook_rejects_negative_counts():
    with pytest.raises(binding.PkvError):
        binding.set_wait_fault(0, -1)


def test_timed_out_wait_tensor_memory_path():
    # The E4M3 decode runs its products on the tensor cores and holds tensor
    # memory per CTA. A timed-out wait frees it on the way out: the next calls,
    # with more CTAs than SMs (CTAs of a later wave allocate on SMs that
    # earlier CTAs left), complete and match the oracle.
    spec = W.WorkloadSpec("timeout_e4m3", 6, 32, 8, 128, 16, "bf16", 1.0)
    lengths = [700, 65, 2049, 1, 300, 1500]
    st, v = W.make_workload(spec, seed=42, lengths=lengths)
    kp, vp = v["k_pool"].clone(), v["v_pool"].clone()
    oracle.append(v["k_new"], v["v_new"], st.slot_mapping, kp, vp)
    NB, Hk, B, D = kp.shape
    slots = []
    for s, L in enumerate(lengths):
        slots += [int(st.block_tables[s, t // B]) * B + t % B for t in range(L)]
    sl = torch.tensor(slots, dtype=torch.int64)
    kr, vr = kp[sl // B, :, sl % B].contiguous(), vp[sl // B, :, sl % B].contiguous()

    def pools(dev):
        kc = torch.full((NB, Hk, B, D), 0x7F, dtype=torch.uint8, device=dev)
        ks = torch.full((NB, Hk, B), float("nan"), dtype=torch.float32, device=dev)
        return kc, kc.clone(), ks, ks.clone()

    ref = pools("cpu")
    oracle.append_quant("fp8_e4m3", kr, vr, sl, *ref)
    cache = binding.QuantCache(*pools("cuda"), "fp8_e4m3", kr.dtype)
    binding.append_quant(kr.cuda(), vr.cuda(), sl.cuda(), cache)
    scale = 1.0 / math.sqrt(128)
    want = oracle.decode_quant("fp8_e4m3", v["q"], *ref, st.block_tables, st.context_lens, scale)
    q, bt, cl = v["q"].cuda(), st.block_tables.cuda(), st.context_lens.cuda()
    torch.cuda.synchronize()
    assert binding.get_error() == 0
    ws = binding.alloc_quant_workspace(cache, 32, 0)
    binding.set_wait_fault(SHORT_NS, 1)
    try:
        binding.decode_attention_quant(q, cache, bt, cl, scale, out_dtype=torch.float32,
                                       workspace=ws)
        status, word = binding.get_error_status()
    finally:
        binding.set_wait_fault(0, 0)
    assert status == PKV_ERR_TIMEOUT and word & binding.DEVERR_TIMEOUT
    for C in (0, 500):
        ws = binding.alloc_quant_workspace(cache, 32, C)
        out = binding.decode_attention_quant(q, cache, bt, cl, scale, out_dtype=torch.float32,
                                             workspace=ws, num_ctas=C)
        assert binding.get_error_status() == (0, 0)
        assert _err(out, want) <= 2e-3
