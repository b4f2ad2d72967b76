"""CPU checks of the C ABI: the library builds, loads and exports every entry
point include/pkv.h declares; host-side argument checks reject bad calls
before touching a GPU; the split-K decomposition is consistent."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from paged_kv_cache_47_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("pkv.h", "pkv_block_manager.h", "pkv_flat.h")]


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.lib()


def declared_functions():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (pkv_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert L.pkv_status_string(code) not in (b"", b"unknown status")
    assert L.pkv_status_string(-99) == b"unknown status"


def _desc(nb=8, b=16, hk=2, d=64, dt=binding.PKV_BF16):
    return binding.CacheDesc(nb, b, hk, d, dt)


def _append(L, desc, kn=16, vn=16, sm=16, n=1, kp=16, vp=16):
    return L.pkv_append(ctypes.byref(desc) if desc is not None else None, kn, vn, sm, n, kp, vp,
                        None)


def test_append_rejects_bad_arguments(L):
    assert _append(L, None) == -1
    assert _append(L, _desc(dt=7)) == -2
    assert _append(L, _desc(b=12)) == -2
    assert _append(L, _desc(d=96)) == -2
    assert _append(L, _desc(hk=0)) == -1
    assert _append(L, _desc(nb=0)) == -1
    assert _append(L, _desc(), n=-1) == -1
    assert _append(L, _desc(), n=0) == 0           # no-op
    assert _append(L, _desc(), kn=None) == -1
    assert _append(L, _desc(), kp=24) == -1        # misaligned
    assert b"aligned" in L.pkv_last_error_message()


def test_append_ex_checks_like_append(L):
    # the options change only when the inputs are read, not what is accepted
    opts = binding.AppendOptions(1)
    d = _desc()

    def call(desc, n=4, kn=16, kp=16, o=opts):
        return L.pkv_append_ex(ctypes.byref(desc) if desc is not None else None, kn, 16, 16, n,
                               kp, 16, None, ctypes.byref(o) if o is not None else None)
    assert call(None) == -1
    assert call(_desc(dt=7)) == -2
    assert call(d, n=-1) == -1
    assert call(d, n=0) == 0                       # no-op
    assert call(d, n=0, o=None) == 0               # NULL options: the defaults
    assert call(d, kn=None) == -1
    assert call(d, kp=24) == -1                    # misaligned


def _decode(L, desc, S=1, Hq=4, q=16, kp=16, vp=16, bt=16, M=4, cl=16, scale=1.0, out=16,
            odt=2, ws=16, wsb=1 << 30, opts=None):
    return L.pkv_decode_attention_ex(ctypes.byref(desc), q, S, Hq, kp, vp, bt, M, cl, scale,
                                     out, odt, ws, wsb, None,
                                     ctypes.byref(opts) if opts is not None else None)


def test_decode_rejects_bad_arguments(L):
    d = _desc()
    assert _decode(L, d, Hq=3) == -1                       # Hq % Hk
    assert _decode(L, d, S=-1) == -1
    assert _decode(L, d, odt=5) == -2
    assert _decode(L, d, M=0) == -1
    assert _decode(L, d, scale=float("nan")) == -1
    o = binding.DecodeOptions()
    o.consumer = 2
    assert _decode(L, _desc(dt=binding.PKV_F32), opts=o) == -2   # mma needs 16-bit
    o.consumer = 3
    assert _decode(L, d, opts=o) == -1
    o.consumer = 0
    o.num_ctas = 4097                                      # above PKV_MAX_DECODE_CTAS
    assert _decode(L, d, opts=o) == -1
    o.num_ctas = -1
    assert _decode(L, d, opts=o) == -1
    assert _decode(L, d, S=0) == 0                         # no-op
    assert _decode(L, d, q=None) == -1
    assert _decode(L, d, q=8) == -1                        # misaligned q
    o.num_ctas = 4
    o.pending_tail = -1
    assert _decode(L, d, opts=o) == -1
    assert b"pending_tail" in L.pkv_last_error_message()
    o.pending_tail = 1                                     # needs tables_ready
    assert _decode(L, d, opts=o) == -1
    assert b"tables_ready" in L.pkv_last_error_message()


def _qdesc(nb=8, b=16, hk=2, d=128, code=binding.PKV_INT8, act=binding.PKV_BF16):
    return binding.QCacheDesc(nb, b, hk, d, code, act)


def _qdecode(L, desc, S=1, Hq=4, q=16, kc=16, vc=16, ks=16, vs=16, opts=None):
    return L.pkv_decode_attention_quant(ctypes.byref(desc), q, S, Hq, kc, vc, ks, vs, 16, 4, 16,
                                        1.0, 16, 2, 16, 1 << 30, None,
                                        ctypes.byref(opts) if opts is not None else None)


def test_quant_calls_reject_bad_arguments(L):
    assert _qdecode(L, _qdesc(code=binding.PKV_BF16)) == -2        # not a code dtype
    assert _qdecode(L, _qdesc(act=binding.PKV_F32)) == -2          # activations 16-bit only
    assert _qdecode(L, _qdesc(d=64)) == -2                         # head_dim 128 only
    assert _qdecode(L, _qdesc(b=12)) == -2
    assert _qdecode(L, _qdesc(), Hq=3) == -1
    o = binding.DecodeOptions()
    o.consumer = 1
    assert _qdecode(L, _qdesc(), opts=o) == -2                    # CUDA-core math: not for codes
    assert _qdecode(L, _qdesc(), ks=None) == -1
    assert _qdecode(L, _qdesc(), vs=8) == -1                       # misaligned scales
    assert _qdecode(L, _qdesc(), S=0) == 0
    d = _qdesc()
    assert L.pkv_append_quant(ctypes.byref(d), 16, 16, 16, 1, 16, 16, None, 16, None) == -1
    assert L.pkv_append_quant(ctypes.byref(d), 16, 16, 16, 1, 16, 16, 8, 16, None) == -1
    assert L.pkv_append_quant(ctypes.byref(d), 16, 16, 16, 0, 16, 16, 16, 16, None) == 0
    p = torch.tensor([[0, 8]], dtype=torch.int64)
    assert L.pkv_block_copy_quant(ctypes.byref(d), p.data_ptr(), 1, 16, 16, 16, 16, None) == -1
    assert L.pkv_block_copy_quant(ctypes.byref(d), p.data_ptr(), 1, 16, 16, None, 16, None) == -1


def test_quant_workspace_formula(L):
    d = _qdesc(hk=8)
    cnt = 4096 * 16
    assert L.pkv_decode_quant_workspace_bytes(ctypes.byref(d), 32, 10) == cnt + 10 * 2 * 4 * 132 * 4
    assert L.pkv_decode_quant_workspace_bytes(ctypes.byref(d), 33, 10) == 0
    assert L.pkv_decode_quant_workspace_bytes(ctypes.byref(_qdesc(d=64)), 32, 10) == 0


def test_block_copy_rejects_bad_pairs(L):
    d = _desc(nb=10)

    def call(pairs):
        p = torch.tensor(pairs, dtype=torch.int64)
        return L.pkv_block_copy(ctypes.byref(d), p.data_ptr(), p.shape[0], 16, 16, None)

    assert call([[0, 10]]) == -1          # out of range
    assert call([[-1, 3]]) == -1
    assert call([[1, 2], [3, 2]]) == -1   # same destination twice
    assert call([[1, 2], [2, 3]]) == -1   # a destination that is also a source
    assert L.pkv_block_copy(ctypes.byref(d), None, 1, 16, 16, None) == -1
    assert L.pkv_block_copy(ctypes.byref(d), None, 0, 16, 16, None) == 0


def test_workspace_size_formula(L):
    d = _desc(hk=8, d=128)
    # 4096 CTAs x 4 arrival counters x 4 bytes, then C CTAs x 2 slots x
    # heads-per-unit x (D outputs + 4 per-warp lse copies) x 4 bytes
    cnt = 4096 * 16
    assert L.pkv_decode_workspace_bytes_ex(ctypes.byref(d), 32, 10) == cnt + 10 * 2 * 4 * 132 * 4
    assert L.pkv_decode_workspace_bytes_ex(ctypes.byref(d), 8 * 40, 3) == cnt + 3 * 2 * 16 * 132 * 4
    assert L.pkv_decode_workspace_bytes_ex(ctypes.byref(d), 32, 4097) == 0
    assert L.pkv_decode_workspace_bytes_ex(ctypes.byref(d), 33, 10) == 0


def test_decomposition_exhaustive(tmp_path):
    exe = tmp_path / "decomp_check"
    subprocess.run(["g++", "-O2", "-std=c++17", "-I", os.path.join(ROOT, "paged_kv_cache_47_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "decomp_check.cpp"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout
