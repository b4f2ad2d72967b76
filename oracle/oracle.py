"""ctypes wrapper over the C oracle — test infrastructure only.

Marshals CPU torch tensors to the C functions in pkv_oracle.c; it computes
nothing itself. Tensors must be contiguous CPU tensors in the layouts of the C
file's header: q [S][Hq][D], pools [NB][Hk][B][D], block_tables [S][M] int32,
context_lens [S] int32, slot_mapping [N] int64, pairs [n][2] int64.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np
import torch

from . import build_oracle

_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        L = ctypes.CDLL(path)
        vp, i32, i64p, i32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        L.oracle_decode.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, i32, i32p, i32,
                                    i32p, ctypes.c_double, vp]
        L.oracle_decode.restype = i32
        L.oracle_append.argtypes = [vp, vp, i64p, i32, vp, vp, i32, i32, i32, i32, i32]
        L.oracle_append.restype = i32
        L.oracle_block_copy.argtypes = [i64p, i32, vp, vp, i32, i32, i32, i32, i32]
        L.oracle_block_copy.restype = i32
        L.oracle_decode_elem.argtypes = [i32, ctypes.c_uint32]
        L.oracle_decode_elem.restype = ctypes.c_double
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = i32
        L.oracle_append_quant.argtypes = [i32, i32, vp, vp, i64p, i32, vp, vp, vp, vp, i32, i32,
                                          i32, i32]
        L.oracle_append_quant.restype = i32
        L.oracle_decode_quant.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp,
                                          i32, i32p, i32, i32p, ctypes.c_double, vp]
        L.oracle_decode_quant.restype = i32
        L.oracle_e4m3_decode.argtypes = [i32]
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = i32
        L.oracle_decode_flat.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, i32, i32p,
                                         i32p, ctypes.c_double, vp]
        L.oracle_decode_flat.restype = i32
        L.oracle_set_num_threads.argtypes = [i32]
        L.oracle_set_num_threads.restype = None
        _lib = L
    return _lib


def _cpu(t: torch.Tensor) -> torch.Tensor:
    assert t.device.type == "cpu", "the oracle takes CPU tensors"
    return t.contiguous()


def decode(q, k_pool, v_pool, block_tables, context_lens, scale: float,
           seq_ids: Optional[Sequence[int]] = None) -> np.ndarray:
    """fp64 attention output [S'][Hq][D] for the sequences `seq_ids` (all if None)."""
    q, k_pool, v_pool = _cpu(q), _cpu(k_pool), _cpu(v_pool)
    bt, cl = _cpu(block_tables).to(torch.int32), _cpu(context_lens).to(torch.int32)
    if seq_ids is not None:
        idx = torch.as_tensor(list(seq_ids), dtype=torch.long)
        q, bt, cl = q[idx].contiguous(), bt[idx].contiguous(), cl[idx].contiguous()
    assert q.dtype == k_pool.dtype == v_pool.dtype
    S, Hq, D = q.shape
    NB, Hk, B, D2 = k_pool.shape
    assert D2 == D
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = lib().oracle_decode(q.data_ptr(), _CODES[q.dtype], S, Hq, Hk, D, B,
                             k_pool.data_ptr(), v_pool.data_ptr(), NB,
                             bt.data_ptr(), bt.shape[1], cl.data_ptr(), float(scale),
                             out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_decode failed with status {rc}")
    return out


def append(k_new, v_new, slot_mapping, k_pool, v_pool) -> None:
    """In-place slot write of one K/V row per token into CPU pools."""
    assert k_pool.is_contiguous() and v_pool.is_contiguous()
    k_new, v_new = _cpu(k_new), _cpu(v_new)
    sm = _cpu(slot_mapping).to(torch.int64)
    NB, Hk, B, D = k_pool.shape
    rc = lib().oracle_append(k_new.data_ptr(), v_new.data_ptr(), sm.data_ptr(), sm.numel(),
                             k_pool.data_ptr(), v_pool.data_ptr(), _CODES[k_pool.dtype],
                             NB, Hk, B, D)
    if rc != 0:
        raise ValueError(f"oracle_append failed with status {rc}")


def block_copy(pairs, k_pool, v_pool) -> None:
    """In-place whole-block copy (src -> dst) in CPU pools."""
    assert k_pool.is_contiguous() and v_pool.is_contiguous()
    p = _cpu(torch.as_tensor(pairs, dtype=torch.int64).reshape(-1, 2))
    NB, Hk, B, D = k_pool.shape
    rc = lib().oracle_block_copy(p.data_ptr(), p.shape[0], k_pool.data_ptr(), v_pool.data_ptr(),
                                 _CODES[k_pool.dtype], NB, Hk, B, D)
    if rc != 0:
        raise ValueError(f"oracle_block_copy failed with status {rc}")


def decode_elem(dtype: torch.dtype, bits: int) -> float:
    return lib().oracle_decode_elem(_CODES[dtype], bits)


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of later oracle calls (OpenMP); n >= 1."""
    lib().oracle_set_num_threads(int(n))


# ------------------------------------------------------------------ quantized KV
QUANT_KINDS = {"int8": 1, "fp8_e4m3": 2}


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (NaN for the two NaN codes)."""
    return lib().oracle_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code of an fp32 value (ties to even, saturating at 448)."""
    return lib().oracle_e4m3_encode(float(x))


def append_quant(kind: str, k_new, v_new, slot_mapping, k_codes, v_codes, k_scales, v_scales):
    """In-place quantized append: k_new/v_new [N][Hk][D] (fp16/bf16) into code
    pools [NB][Hk][B][D] (uint8) and scale pools [NB][Hk][B] (fp32)."""
    for t in (k_codes, v_codes, k_scales, v_scales):
        assert t.is_contiguous() and t.device.type == "cpu"
    assert k_codes.dtype == v_codes.dtype == torch.uint8
    assert k_scales.dtype == v_scales.dtype == torch.float32
    k_new, v_new = _cpu(k_new), _cpu(v_new)
    assert k_new.dtype == v_new.dtype and k_new.dtype in (torch.float16, torch.bfloat16)
    sm = _cpu(slot_mapping).to(torch.int64)
    NB, Hk, B, D = k_codes.shape
    rc = lib().oracle_append_quant(QUANT_KINDS[kind], _CODES[k_new.dtype], k_new.data_ptr(),
                                   v_new.data_ptr(), sm.data_ptr(), sm.numel(),
                                   k_codes.data_ptr(), v_codes.data_ptr(), k_scales.data_ptr(),
                                   v_scales.data_ptr(), NB, Hk, B, D)
    if rc != 0:
        raise ValueError(f"oracle_append_quant failed with status {rc}")


def decode_quant(kind: str, q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                 scale: float, seq_ids: Optional[Sequence[int]] = None) -> np.ndarray:
    """fp64 attention output [S'][Hq][D] over a quantized cache."""
    q = _cpu(q)
    kc, vc, ks, vs = _cpu(k_codes), _cpu(v_codes), _cpu(k_scales), _cpu(v_scales)
    bt, cl = _cpu(block_tables).to(torch.int32), _cpu(context_lens).to(torch.int32)
    if seq_ids is not None:
        idx = torch.as_tensor(list(seq_ids), dtype=torch.long)
        q, bt, cl = q[idx].contiguous(), bt[idx].contiguous(), cl[idx].contiguous()
    assert q.dtype in (torch.float16, torch.bfloat16)
    S, Hq, D = q.shape
    NB, Hk, B, D2 = kc.shape
    assert D2 == D and ks.shape == (NB, Hk, B)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = lib().oracle_decode_quant(q.data_ptr(), _CODES[q.dtype], S, Hq, Hk, D, B,
                                   QUANT_KINDS[kind], kc.data_ptr(), vc.data_ptr(), ks.data_ptr(),
                                   vs.data_ptr(), NB, bt.data_ptr(), bt.shape[1], cl.data_ptr(),
                                   float(scale), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_decode_quant failed with status {rc}")
    return out


# ------------------------------------------------------------------ flat spans
def decode_flat(q, k_flat, v_flat, slots, context_lens, scale: float) -> np.ndarray:
    """fp64 attention output [S][Hq][D]; sequence s reads span slots[s] of
    k_flat / v_flat [num_slots][capacity][Hk][D] (token-major)."""
    q, kf, vf = _cpu(q), _cpu(k_flat), _cpu(v_flat)
    sl = _cpu(torch.as_tensor(slots)).to(torch.int32)
    cl = _cpu(context_lens).to(torch.int32)
    assert q.dtype == kf.dtype == vf.dtype and kf.shape == vf.shape
    S, Hq, D = q.shape
    NS, cap, Hk, D2 = kf.shape
    assert D2 == D
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = lib().oracle_decode_flat(q.data_ptr(), _CODES[q.dtype], S, Hq, Hk, D, kf.data_ptr(),
                                  vf.data_ptr(), NS, cap, sl.data_ptr(), cl.data_ptr(),
                                  float(scale), out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_decode_flat failed with status {rc}")
    return out
