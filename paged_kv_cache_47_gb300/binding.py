"""Python binding over libpkv's C ABI (include/pkv.h).

Argument marshalling only: every step of the hot path runs in libpkv's CUDA
kernels. There is no CPU fallback; if the library is missing or a call fails,
these functions raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

PKV_F32, PKV_F16, PKV_BF16, PKV_INT8, PKV_FP8_E4M3 = 0, 1, 2, 3, 4
CODE_DTYPES = {"int8": PKV_INT8, "fp8_e4m3": PKV_FP8_E4M3}
DTYPE_CODE = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}
CODE_DTYPE = {v: k for k, v in DTYPE_CODE.items()}

STATUS = {0: "PKV_OK", -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_UNSUPPORTED", -3: "PKV_ERR_CUDA",
          -4: "PKV_ERR_OUT_OF_RANGE", -5: "PKV_ERR_TIMEOUT", -6: "PKV_ERR_WORKSPACE"}
DEVERR_BLOCK_ID, DEVERR_CONTEXT, DEVERR_TIMEOUT, DEVERR_SLOT = 0x1, 0x2, 0x4, 0x8


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class QCacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("code_dtype", ctypes.c_int32), ("act_dtype", ctypes.c_int32)]


class DecodeOptions(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int32), ("consumer", ctypes.c_int32),
                ("timing_events", ctypes.c_void_p * 2), ("lse_out", ctypes.c_void_p),
                ("tables_ready", ctypes.c_int32), ("pending_tail", ctypes.c_int32)]


class PreparedBmStep:
    """pkv_bm_append_batch + pkv_bm_block_tables for a fixed batch of sequences,
    marshalled once: each call reuses the same host buffers, so what remains per
    step is the two native calls. The returned tensors are views of those
    buffers, overwritten by the next call."""

    def __init__(self, bm, seq_ids, num_tokens, max_blocks_per_seq: int):
        self._ids = torch.as_tensor(list(seq_ids), dtype=torch.int64).contiguous()
        self._nt = torch.as_tensor(list(num_tokens), dtype=torch.int32).contiguous()
        S = len(self._ids)
        self._total = int(self._nt.sum()) if S else 0
        self.slots = torch.empty(max(1, self._total), dtype=torch.int64)
        self.pairs = torch.empty(max(1, S), 2, dtype=torch.int64)
        self.tables = torch.empty(S, max_blocks_per_seq, dtype=torch.int32)
        self.lens = torch.empty(S, dtype=torch.int32)
        self._nc, self._nd = ctypes.c_int32(0), ctypes.c_int32(0)
        L, h = bm._L, bm._h
        self._bm = bm       # keeps the manager alive
        self._append = (L.pkv_bm_append_batch,
                        (h, self._ids.data_ptr(), self._nt.data_ptr(), S, self.slots.data_ptr(),
                         self.pairs.data_ptr(), S, ctypes.byref(self._nc),
                         ctypes.byref(self._nd)))
        self._tables = (L.pkv_bm_block_tables,
                        (h, self._ids.data_ptr(), S, max_blocks_per_seq, self.tables.data_ptr(),
                         self.lens.data_ptr()))
        self._slots_view = self.slots[:self._total]
        self._no_pairs = self.pairs[:0]

    def append(self):
        """(slots, copy pairs) of the step's new tokens."""
        fn, args = self._append
        _bm_check(fn(*args))
        nc = self._nc.value
        return self._slots_view, (self.pairs[:nc] if nc else self._no_pairs)

    def block_tables(self):
        """(block_tables [S][M], context_lens [S]) of the batch."""
        fn, args = self._tables
        _bm_check(fn(*args))
        return self.tables, self.lens


class AppendOptions(ctypes.Structure):
    _fields_ = [("inputs_ready", ctypes.c_int32)]


class PrefixGroups(ctypes.Structure):
    _fields_ = [("num_groups", ctypes.c_int32), ("group_of_seq", ctypes.c_void_p),
                ("group_prefix_blocks", ctypes.c_void_p)]


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load libpkv (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libpkv is not built ({path}); run paged_kv_cache_47_gb300.build.build()")
        L = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        dp = ctypes.POINTER(CacheDesc)
        L.pkv_append.argtypes = [dp, vp, vp, vp, i32, vp, vp, vp]
        L.pkv_append.restype = i32
        L.pkv_append_ex.argtypes = [dp, vp, vp, vp, i32, vp, vp, vp,
                                    ctypes.POINTER(AppendOptions)]
        L.pkv_append_ex.restype = i32
        L.pkv_decode_workspace_bytes.argtypes = [dp, i32, i32, i32]
        L.pkv_decode_workspace_bytes.restype = sz
        L.pkv_decode_workspace_bytes_ex.argtypes = [dp, i32, i32]
        L.pkv_decode_workspace_bytes_ex.restype = sz
        dec = [dp, vp, i32, i32, vp, vp, vp, i32, vp, ctypes.c_float, vp, i32, vp, sz, vp]
        L.pkv_decode_attention.argtypes = dec
        L.pkv_decode_attention.restype = i32
        L.pkv_decode_attention_ex.argtypes = dec + [ctypes.POINTER(DecodeOptions)]
        L.pkv_decode_attention_ex.restype = i32
        L.pkv_append_decode_attention.argtypes = [dp, vp, i32, i32, vp, vp, vp, vp, vp, i32, vp,
                                                  ctypes.c_float, vp, i32, vp, sz, vp,
                                                  ctypes.POINTER(DecodeOptions)]
        L.pkv_append_decode_attention.restype = i32
        L.pkv_block_copy.argtypes = [dp, vp, i32, vp, vp, vp]
        L.pkv_block_copy.restype = i32
        qp = ctypes.POINTER(QCacheDesc)
        L.pkv_append_quant.argtypes = [qp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
        L.pkv_append_quant.restype = i32
        L.pkv_append_quant_ex.argtypes = [qp, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                          ctypes.POINTER(AppendOptions)]
        L.pkv_append_quant_ex.restype = i32
        L.pkv_decode_quant_workspace_bytes.argtypes = [qp, i32, i32]
        L.pkv_decode_quant_workspace_bytes.restype = sz
        L.pkv_decode_attention_quant.argtypes = [qp, vp, i32, i32, vp, vp, vp, vp, vp, i32, vp,
                                                 ctypes.c_float, vp, i32, vp, sz, vp,
                                                 ctypes.POINTER(DecodeOptions)]
        L.pkv_decode_attention_quant.restype = i32
        L.pkv_append_decode_attention_quant.argtypes = [qp, vp, i32, i32, vp, vp, vp, vp, vp, vp,
                                                        vp, i32, vp, ctypes.c_float, vp, i32, vp,
                                                        sz, vp, ctypes.POINTER(DecodeOptions)]
        L.pkv_append_decode_attention_quant.restype = i32
        L.pkv_block_copy_quant.argtypes = [qp, vp, i32, vp, vp, vp, vp, vp]
        L.pkv_block_copy_quant.restype = i32
        L.pkv_decode_prefix_workspace_bytes.argtypes = [dp, i32, i32, i32,
                                                        ctypes.POINTER(PrefixGroups), i32]
        L.pkv_decode_prefix_workspace_bytes.restype = sz
        L.pkv_decode_attention_prefix.argtypes = [dp, vp, i32, i32, vp, vp, vp, i32, vp,
                                                  ctypes.c_float, ctypes.POINTER(PrefixGroups),
                                                  vp, i32, vp, sz, vp,
                                                  ctypes.POINTER(DecodeOptions)]
        L.pkv_decode_attention_prefix.restype = i32
        L.pkv_debug_set_wait_fault.argtypes = [ctypes.c_uint64, i32]
        L.pkv_debug_set_wait_fault.restype = i32
        L.pkv_get_error.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
        L.pkv_get_error.restype = i32
        L.pkv_status_string.argtypes = [i32]
        L.pkv_status_string.restype = ctypes.c_char_p
        L.pkv_last_error_message.argtypes = []
        L.pkv_last_error_message.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise PkvError(status, lib().pkv_last_error_message().decode())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def cache_desc(k_pool: torch.Tensor) -> CacheDesc:
    """Descriptor of a pool tensor [NB][Hk][B][D]."""
    NB, Hk, B, D = k_pool.shape
    return CacheDesc(NB, B, Hk, D, DTYPE_CODE[k_pool.dtype])


def _pools(k_pool, v_pool):
    if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype:
        raise ValueError("k_pool and v_pool differ in shape or dtype")
    if not (k_pool.is_contiguous() and v_pool.is_contiguous()):
        raise ValueError("pools must be contiguous")
    return cache_desc(k_pool)


def append(k_new, v_new, slot_mapping, k_pool, v_pool, stream=None,
           inputs_ready: bool = False) -> None:
    """Write k_new/v_new [N][Hk][D] into the pools at slot_mapping [N] (int64).
    inputs_ready: no kernel that may still be running writes the three inputs, so
    they are read before the wait on the preceding kernel (pkv_append_options)."""
    desc = _pools(k_pool, v_pool)
    k_new, v_new = k_new.contiguous(), v_new.contiguous()
    sm = slot_mapping.contiguous()
    assert sm.dtype == torch.int64 and k_new.dtype == k_pool.dtype
    opts = AppendOptions(int(inputs_ready))
    _check(lib().pkv_append_ex(ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(sm),
                               sm.numel(), _ptr(k_pool), _ptr(v_pool), _stream(stream),
                               ctypes.byref(opts)))


def workspace_bytes(k_pool, num_q_heads: int, num_ctas: int = 0) -> int:
    desc = cache_desc(k_pool)
    return int(lib().pkv_decode_workspace_bytes_ex(ctypes.byref(desc), num_q_heads, num_ctas))


def alloc_workspace(k_pool, num_q_heads: int, num_ctas: int = 0) -> torch.Tensor:
    """Split-K workspace, zero-filled as the library requires before first use
    (its arrival counters; every call leaves them zero again)."""
    n = workspace_bytes(k_pool, num_q_heads, num_ctas)
    if n == 0:
        raise PkvError(-1, "workspace size query failed")
    return torch.zeros(n, dtype=torch.uint8, device=k_pool.device)


def decode_attention(q, k_pool, v_pool, block_tables, context_lens, scale: float,
                     out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
                     workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                     consumer: int = 0, timing_events: Optional[Sequence] = None,
                     stream=None, lse_out: Optional[torch.Tensor] = None,
                     tables_ready: bool = False, pending_tail: int = 0) -> torch.Tensor:
    """Paged decode attention: out[s][h] = softmax(scale q K^T) V over context_lens[s] tokens.
    tables_ready: the caller promises that no kernel that may still be running writes the
    tables or lengths (pkv_decode_options.tables_ready).
    pending_tail: n > 0 promises, besides, that no kernel that may still be running
    writes q or any row below the last n of each sequence
    (pkv_decode_options.pending_tail)."""
    desc = _pools(k_pool, v_pool)
    S, Hq, D = q.shape
    q = q.contiguous()
    bt = block_tables.contiguous()
    cl = context_lens.contiguous()
    assert bt.dtype == torch.int32 and cl.dtype == torch.int32 and q.dtype == k_pool.dtype
    if out is None:
        out = torch.empty(S, Hq, D, dtype=out_dtype or q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(k_pool, Hq, num_ctas)
    opts = DecodeOptions()
    opts.num_ctas = num_ctas
    opts.consumer = consumer
    opts.tables_ready = int(tables_ready)
    opts.pending_tail = int(pending_tail)
    if timing_events is not None:
        for i, ev in enumerate(timing_events):
            opts.timing_events[i] = None if ev is None else ev.cuda_event
    if lse_out is not None:
        assert lse_out.dtype == torch.float32 and lse_out.shape == (S, Hq) and lse_out.is_contiguous()
        opts.lse_out = lse_out.data_ptr()
    _check(lib().pkv_decode_attention_ex(
        ctypes.byref(desc), _ptr(q), S, Hq, _ptr(k_pool), _ptr(v_pool), _ptr(bt), bt.shape[1],
        _ptr(cl), float(scale), _ptr(out), DTYPE_CODE[out.dtype], _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream), ctypes.byref(opts)))
    return out


class PreparedDecode:
    """A decode-attention call whose arguments are marshalled once.

    For repeated decode steps on stable buffers (the usual serving loop, and
    CUDA-graph capture): the tensors' addresses, shapes and the workspace are
    fixed at construction; each call only passes the stream. The caller keeps
    the tensors alive and rewrites their contents in place between steps.
    """

    def __init__(self, q, k_pool, v_pool, block_tables, context_lens, scale: float,
                 out: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                 num_ctas: int = 0, consumer: int = 0, tables_ready: bool = False,
                 pending_tail: int = 0):
        self._desc = _pools(k_pool, v_pool)
        for t in (q, block_tables, context_lens, out):
            if not t.is_contiguous():
                raise ValueError("prepared decode needs contiguous tensors")
        assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
        assert q.dtype == k_pool.dtype
        S, Hq, D = q.shape
        if workspace is None:
            workspace = alloc_workspace(k_pool, Hq, num_ctas)
        self._keep = (q, k_pool, v_pool, block_tables, context_lens, out, workspace)
        self._opts = DecodeOptions()
        self._opts.num_ctas = num_ctas
        self._opts.consumer = consumer
        self._opts.tables_ready = int(tables_ready)
        self._opts.pending_tail = int(pending_tail)
        self._args = (ctypes.byref(self._desc), q.data_ptr(), S, Hq, k_pool.data_ptr(),
                      v_pool.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                      context_lens.data_ptr(), float(scale), out.data_ptr(),
                      DTYPE_CODE[out.dtype], workspace.data_ptr(),
                      workspace.numel() * workspace.element_size())
        self._fn = lib().pkv_decode_attention_ex
        self.out = out

    def __call__(self, stream, timing_events: Optional[Sequence] = None) -> None:
        opts = self._opts
        for i in range(2):
            ev = timing_events[i] if timing_events is not None else None
            opts.timing_events[i] = None if ev is None else ev.cuda_event
        _check(self._fn(*self._args, _stream(stream), ctypes.byref(opts)))


def append_decode_attention(q, k_new, v_new, k_pool, v_pool, block_tables, context_lens,
                            scale: float, out: Optional[torch.Tensor] = None,
                            out_dtype: Optional[torch.dtype] = None,
                            workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                            consumer: int = 0, stream=None, tables_ready: bool = False,
                            pending_tail: int = 0) -> torch.Tensor:
    """One decode step in one launch (pkv_append_decode_attention): each
    sequence's new row k_new[s] / v_new[s] [S][Hk][D] goes to position
    context_lens[s] - 1 (the slot its block table gives), and the attention
    runs over the context including it."""
    desc = _pools(k_pool, v_pool)
    S, Hq, D = q.shape
    q, k_new, v_new = q.contiguous(), k_new.contiguous(), v_new.contiguous()
    bt, cl = block_tables.contiguous(), context_lens.contiguous()
    assert bt.dtype == torch.int32 and cl.dtype == torch.int32
    assert q.dtype == k_pool.dtype == k_new.dtype == v_new.dtype
    if out is None:
        out = torch.empty(S, Hq, D, dtype=out_dtype or q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(k_pool, Hq, num_ctas)
    opts = DecodeOptions()
    opts.num_ctas = num_ctas
    opts.consumer = consumer
    opts.tables_ready = int(tables_ready)
    opts.pending_tail = int(pending_tail)
    _check(lib().pkv_append_decode_attention(
        ctypes.byref(desc), _ptr(q), S, Hq, _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
        _ptr(bt), bt.shape[1], _ptr(cl), float(scale), _ptr(out), DTYPE_CODE[out.dtype],
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream),
        ctypes.byref(opts)))
    return out


class PreparedAppendDecode(PreparedDecode):
    """A pkv_append_decode_attention call whose arguments are marshalled once
    (see PreparedDecode); k_new and v_new are rewritten in place each step."""

    def __init__(self, q, k_new, v_new, k_pool, v_pool, block_tables, context_lens,
                 scale: float, out: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                 num_ctas: int = 0, consumer: int = 0, tables_ready: bool = False,
                 pending_tail: int = 0):
        super().__init__(q, k_pool, v_pool, block_tables, context_lens, scale, out, workspace,
                         num_ctas, consumer, tables_ready, pending_tail)
        for t in (k_new, v_new):
            if not t.is_contiguous() or t.dtype != k_pool.dtype:
                raise ValueError("k_new / v_new must be contiguous, in the cache dtype")
        self._keep = self._keep + (k_new, v_new)
        a = self._args
        # q, S, Hq | k_new, v_new | pools, tables, ...
        self._args = a[:4] + (k_new.data_ptr(), v_new.data_ptr()) + a[4:]
        self._fn = lib().pkv_append_decode_attention


class PreparedAppend:
    """An append call whose arguments are marshalled once (see PreparedDecode)."""

    def __init__(self, k_new, v_new, slot_mapping, k_pool, v_pool, inputs_ready: bool = False):
        self._desc = _pools(k_pool, v_pool)
        for t in (k_new, v_new, slot_mapping):
            if not t.is_contiguous():
                raise ValueError("prepared append needs contiguous tensors")
        assert slot_mapping.dtype == torch.int64 and k_new.dtype == k_pool.dtype
        self._keep = (k_new, v_new, slot_mapping, k_pool, v_pool)
        self._opts = AppendOptions(int(inputs_ready))
        self._args = (ctypes.byref(self._desc), k_new.data_ptr(), v_new.data_ptr(),
                      slot_mapping.data_ptr(), slot_mapping.numel(), k_pool.data_ptr(),
                      v_pool.data_ptr())
        self._fn = lib().pkv_append_ex

    def __call__(self, stream) -> None:
        _check(self._fn(*self._args, _stream(stream), ctypes.byref(self._opts)))


def block_copy(pairs, k_pool, v_pool, stream=None) -> None:
    """Copy whole blocks src -> dst; pairs is host data [n][2] (list or CPU tensor)."""
    desc = _pools(k_pool, v_pool)
    p = torch.as_tensor(pairs, dtype=torch.int64).reshape(-1, 2).contiguous()
    assert p.device.type == "cpu", "block-copy pairs are host memory"
    _check(lib().pkv_block_copy(ctypes.byref(desc), _ptr(p), p.shape[0], _ptr(k_pool),
                                _ptr(v_pool), _stream(stream)))


def set_wait_fault(wait_limit_ns: int = 0, drop_arrivals: int = 0) -> None:
    """Test hook (pkv_debug_set_wait_fault): the wait limit of the next decode
    launches (0 = the default 2 s) and how many of them withhold one arrival
    so that a bounded wait runs out. (0, 0) restores normal operation."""
    _check(lib().pkv_debug_set_wait_fault(int(wait_limit_ns), int(drop_arrivals)))


def get_error_status(stream=None):
    """(status, word): pkv_get_error's return code and the device error word
    it read and cleared."""
    w = ctypes.c_int32(0)
    st = lib().pkv_get_error(ctypes.byref(w), _stream(stream))
    return int(st), int(w.value)


def get_error(stream=None) -> int:
    """Synchronise and read+clear the device error word (PKV_DEVERR_* bits)."""
    w = ctypes.c_int32(0)
    lib().pkv_get_error(ctypes.byref(w), _stream(stream))
    return int(w.value)


# ------------------------------------------------------------------ 8-bit caches
class QuantCache:
    """An 8-bit paged KV cache: code pools [NB][Hk][B][D] (uint8) and row-scale
    pools [NB][Hk][B] (fp32) for K and V, with the activation dtype of q,
    k_new and v_new. Holds the tensors; the library owns no memory."""

    def __init__(self, k_codes, v_codes, k_scales, v_scales, code: str, act_dtype: torch.dtype):
        for t in (k_codes, v_codes, k_scales, v_scales):
            if not t.is_contiguous():
                raise ValueError("quantized pools must be contiguous")
        if k_codes.dtype != torch.uint8 or v_codes.shape != k_codes.shape:
            raise ValueError("code pools must be uint8 and of one shape")
        NB, Hk, B, D = k_codes.shape
        if k_scales.dtype != torch.float32 or k_scales.shape != (NB, Hk, B) or \
                v_scales.shape != k_scales.shape:
            raise ValueError("scale pools must be float32 [NB][Hk][B]")
        self.k_codes, self.v_codes, self.k_scales, self.v_scales = k_codes, v_codes, k_scales, v_scales
        self.code, self.act_dtype = code, act_dtype
        self.desc = QCacheDesc(NB, B, Hk, D, CODE_DTYPES[code], DTYPE_CODE[act_dtype])

    @classmethod
    def empty(cls, num_blocks, num_kv_heads, block_size, head_dim, code: str,
              act_dtype: torch.dtype, device="cuda"):
        kc = torch.zeros(num_blocks, num_kv_heads, block_size, head_dim, dtype=torch.uint8,
                         device=device)
        ks = torch.zeros(num_blocks, num_kv_heads, block_size, dtype=torch.float32, device=device)
        return cls(kc, kc.clone(), ks, ks.clone(), code, act_dtype)

    def pointers(self):
        return (self.k_codes.data_ptr(), self.v_codes.data_ptr(), self.k_scales.data_ptr(),
                self.v_scales.data_ptr())


def append_quant(k_new, v_new, slot_mapping, cache: QuantCache, stream=None,
                 inputs_ready: bool = False) -> None:
    """Quantize k_new/v_new [N][Hk][D] (the cache's activation dtype) into their slots
    (inputs_ready: see append)."""
    k_new, v_new = k_new.contiguous(), v_new.contiguous()
    sm = slot_mapping.contiguous()
    assert sm.dtype == torch.int64 and k_new.dtype == cache.act_dtype == v_new.dtype
    opts = AppendOptions(int(inputs_ready))
    _check(lib().pkv_append_quant_ex(ctypes.byref(cache.desc), _ptr(k_new), _ptr(v_new), _ptr(sm),
                                     sm.numel(), *cache.pointers(), _stream(stream),
                                     ctypes.byref(opts)))


def quant_workspace_bytes(cache: QuantCache, num_q_heads: int, num_ctas: int = 0) -> int:
    return int(lib().pkv_decode_quant_workspace_bytes(ctypes.byref(cache.desc), num_q_heads,
                                                      num_ctas))


def alloc_quant_workspace(cache: QuantCache, num_q_heads: int, num_ctas: int = 0) -> torch.Tensor:
    """Zero-filled split-K workspace for pkv_decode_attention_quant."""
    n = quant_workspace_bytes(cache, num_q_heads, num_ctas)
    if n == 0:
        raise PkvError(-1, "workspace size query failed")
    return torch.zeros(n, dtype=torch.uint8, device=cache.k_codes.device)


def decode_attention_quant(q, cache: QuantCache, block_tables, context_lens, scale: float,
                           out: Optional[torch.Tensor] = None,
                           out_dtype: Optional[torch.dtype] = None,
                           workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                           consumer: int = 0, timing_events: Optional[Sequence] = None,
                           stream=None, tables_ready: bool = False,
                           pending_tail: int = 0) -> torch.Tensor:
    """Paged decode attention over an 8-bit cache (tables_ready, pending_tail: see
    decode_attention)."""
    S, Hq, D = q.shape
    q = q.contiguous()
    bt, cl = block_tables.contiguous(), context_lens.contiguous()
    assert bt.dtype == torch.int32 and cl.dtype == torch.int32 and q.dtype == cache.act_dtype
    if out is None:
        out = torch.empty(S, Hq, D, dtype=out_dtype or q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_quant_workspace(cache, Hq, num_ctas)
    opts = DecodeOptions()
    opts.num_ctas = num_ctas
    opts.consumer = consumer
    opts.tables_ready = int(tables_ready)
    opts.pending_tail = int(pending_tail)
    if timing_events is not None:
        for i, ev in enumerate(timing_events):
            opts.timing_events[i] = None if ev is None else ev.cuda_event
    _check(lib().pkv_decode_attention_quant(
        ctypes.byref(cache.desc), _ptr(q), S, Hq, *cache.pointers(), _ptr(bt), bt.shape[1],
        _ptr(cl), float(scale), _ptr(out), DTYPE_CODE[out.dtype], _ptr(workspace),
        workspace.numel(), _stream(stream), ctypes.byref(opts)))
    return out


class PreparedDecodeQuant:
    """pkv_decode_attention_quant with its arguments marshalled once (see PreparedDecode)."""

    def __init__(self, q, cache: QuantCache, block_tables, context_lens, scale: float,
                 out: torch.Tensor, workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                 tables_ready: bool = False, pending_tail: int = 0):
        for t in (q, block_tables, context_lens, out):
            if not t.is_contiguous():
                raise ValueError("prepared decode needs contiguous tensors")
        assert q.dtype == cache.act_dtype
        S, Hq, D = q.shape
        if workspace is None:
            workspace = alloc_quant_workspace(cache, Hq, num_ctas)
        self._keep = (q, cache, block_tables, context_lens, out, workspace)
        self._opts = DecodeOptions()
        self._opts.num_ctas = num_ctas
        self._opts.tables_ready = int(tables_ready)
        self._opts.pending_tail = int(pending_tail)
        self._args = (ctypes.byref(cache.desc), q.data_ptr(), S, Hq, *cache.pointers(),
                      block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(),
                      float(scale), out.data_ptr(), DTYPE_CODE[out.dtype], workspace.data_ptr(),
                      workspace.numel())
        self._fn = lib().pkv_decode_attention_quant
        self.out = out

    def __call__(self, stream, timing_events: Optional[Sequence] = None) -> None:
        opts = self._opts
        for i in range(2):
            ev = timing_events[i] if timing_events is not None else None
            opts.timing_events[i] = None if ev is None else ev.cuda_event
        _check(self._fn(*self._args, _stream(stream), ctypes.byref(opts)))


def append_decode_attention_quant(q, k_new, v_new, cache: QuantCache, block_tables,
                                  context_lens, scale: float, out: Optional[torch.Tensor] = None,
                                  out_dtype: Optional[torch.dtype] = None,
                                  workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                                  stream=None, tables_ready: bool = False,
                                  pending_tail: int = 0) -> torch.Tensor:
    """One decode step over an 8-bit cache (pkv_append_decode_attention_quant):
    each sequence's new row k_new[s] / v_new[s] [S][Hk][D] is quantized into
    position context_lens[s] - 1 of its table row, and the attention runs over
    the context including it."""
    S, Hq, D = q.shape
    q, k_new, v_new = q.contiguous(), k_new.contiguous(), v_new.contiguous()
    bt, cl = block_tables.contiguous(), context_lens.contiguous()
    assert bt.dtype == torch.int32 and cl.dtype == torch.int32
    assert q.dtype == k_new.dtype == v_new.dtype == cache.act_dtype
    if out is None:
        out = torch.empty(S, Hq, D, dtype=out_dtype or q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_quant_workspace(cache, Hq, num_ctas)
    opts = DecodeOptions()
    opts.num_ctas = num_ctas
    opts.tables_ready = int(tables_ready)
    opts.pending_tail = int(pending_tail)
    _check(lib().pkv_append_decode_attention_quant(
        ctypes.byref(cache.desc), _ptr(q), S, Hq, _ptr(k_new), _ptr(v_new), *cache.pointers(),
        _ptr(bt), bt.shape[1], _ptr(cl), float(scale), _ptr(out), DTYPE_CODE[out.dtype],
        _ptr(workspace), workspace.numel(), _stream(stream), ctypes.byref(opts)))
    return out


class PreparedAppendQuant:
    """pkv_append_quant with its arguments marshalled once (see PreparedDecode)."""

    def __init__(self, k_new, v_new, slot_mapping, cache: QuantCache, inputs_ready: bool = False):
        for t in (k_new, v_new, slot_mapping):
            if not t.is_contiguous():
                raise ValueError("prepared append needs contiguous tensors")
        assert slot_mapping.dtype == torch.int64 and k_new.dtype == cache.act_dtype
        self._keep = (k_new, v_new, slot_mapping, cache)
        self._opts = AppendOptions(int(inputs_ready))
        self._args = (ctypes.byref(cache.desc), k_new.data_ptr(), v_new.data_ptr(),
                      slot_mapping.data_ptr(), slot_mapping.numel(), *cache.pointers())
        self._fn = lib().pkv_append_quant_ex

    def __call__(self, stream) -> None:
        _check(self._fn(*self._args, _stream(stream), ctypes.byref(self._opts)))


def block_copy_quant(pairs, cache: QuantCache, stream=None) -> None:
    """Copy whole blocks (codes and scales) src -> dst; pairs is host data [n][2]."""
    p = torch.as_tensor(pairs, dtype=torch.int64).reshape(-1, 2).contiguous()
    assert p.device.type == "cpu", "block-copy pairs are host memory"
    _check(lib().pkv_block_copy_quant(ctypes.byref(cache.desc), _ptr(p), p.shape[0],
                                      *cache.pointers(), _stream(stream)))


# ------------------------------------------------------------------ block manager
class BmStats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("shared_blocks", ctypes.c_int32), ("prefix_entries", ctypes.c_int32),
                ("sequences", ctypes.c_int64), ("tokens", ctypes.c_int64)]


def _bm_lib():
    L = lib()
    if not getattr(L, "_bm_ready", False):
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.pkv_bm_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
        L.pkv_bm_create.restype = i32
        L.pkv_bm_destroy.argtypes = [vp]
        L.pkv_bm_destroy.restype = None
        L.pkv_bm_add_sequence.argtypes = [vp, i64, vp, i32, vp]
        L.pkv_bm_add_sequence.restype = i32
        L.pkv_bm_append.argtypes = [vp, i64, i32, vp, vp, i32, ctypes.POINTER(i32)]
        L.pkv_bm_append.restype = i32
        L.pkv_bm_append_batch.argtypes = [vp, vp, vp, i32, vp, vp, i32, ctypes.POINTER(i32),
                                          ctypes.POINTER(i32)]
        L.pkv_bm_append_batch.restype = i32
        L.pkv_bm_fork.argtypes = [vp, i64, i64]
        L.pkv_bm_fork.restype = i32
        L.pkv_bm_free_sequence.argtypes = [vp, i64]
        L.pkv_bm_free_sequence.restype = i32
        L.pkv_bm_block_tables.argtypes = [vp, vp, i32, i32, vp, vp]
        L.pkv_bm_block_tables.restype = i32
        L.pkv_bm_stats_get.argtypes = [vp, ctypes.POINTER(BmStats)]
        L.pkv_bm_stats_get.restype = i32
        L.pkv_bm_refcount.argtypes = [vp, i32]
        L.pkv_bm_refcount.restype = i32
        L.pkv_bm_simulate_admission.argtypes = [i32, i32, vp, i32, i32, ctypes.POINTER(i32),
                                                ctypes.POINTER(ctypes.c_double)]
        L.pkv_bm_simulate_admission.restype = i32
        L._bm_ready = True
    return L


class NoBlocks(PkvError):
    """The block manager has too few free blocks; the call changed nothing."""


def _bm_check(status: int):
    if status == -7:
        raise NoBlocks(status, lib().pkv_last_error_message().decode())
    _check(status)


class BlockManager:
    """Host block manager of a paged KV cache (libpkv's pkv_bm_* calls)."""

    def __init__(self, num_blocks: int, block_size: int):
        L = _bm_lib()
        h = ctypes.c_void_p()
        _bm_check(L.pkv_bm_create(num_blocks, block_size, ctypes.byref(h)))
        self._h, self._L = h, L
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._L.pkv_bm_destroy(h)
            self._h = None

    def add_sequence(self, seq: int, prefix_hashes=()) -> list:
        hs = (ctypes.c_uint64 * max(1, len(prefix_hashes)))(*[int(x) & (2 ** 64 - 1)
                                                              for x in prefix_hashes])
        hits = (ctypes.c_uint8 * max(1, len(prefix_hashes)))()
        _bm_check(self._L.pkv_bm_add_sequence(self._h, seq, hs, len(prefix_hashes), hits))
        return [bool(hits[i]) for i in range(len(prefix_hashes))]

    def append(self, seq: int, n: int):
        """Slots of n new tokens and the (src, dst) copies to run first."""
        slots = (ctypes.c_int64 * max(1, n))()
        pairs = (ctypes.c_int64 * 2)()
        nc = ctypes.c_int32(0)
        _bm_check(self._L.pkv_bm_append(self._h, seq, n, slots, pairs, 1, ctypes.byref(nc)))
        return [slots[i] for i in range(n)], [(pairs[2 * i], pairs[2 * i + 1])
                                               for i in range(nc.value)]

    def append_batch(self, seq_ids, num_tokens):
        """Slots (all sequences back to back) and copies of one step; raises on
        failure after the sequences before the failing one were applied."""
        ids = torch.as_tensor(list(seq_ids), dtype=torch.int64)
        nt = torch.as_tensor(list(num_tokens), dtype=torch.int32)
        total = int(nt.sum()) if len(nt) else 0
        slots = torch.empty(max(1, total), dtype=torch.int64)
        pairs = torch.empty(max(1, len(ids)), 2, dtype=torch.int64)
        nc, nd = ctypes.c_int32(0), ctypes.c_int32(0)
        _bm_check(self._L.pkv_bm_append_batch(self._h, ids.data_ptr(), nt.data_ptr(), len(ids),
                                              slots.data_ptr(), pairs.data_ptr(), len(ids),
                                              ctypes.byref(nc), ctypes.byref(nd)))
        return slots[:total], pairs[:nc.value]

    def fork(self, parent: int, child: int) -> None:
        _bm_check(self._L.pkv_bm_fork(self._h, parent, child))

    def free_sequence(self, seq: int) -> None:
        _bm_check(self._L.pkv_bm_free_sequence(self._h, seq))

    def block_tables(self, seq_ids, max_blocks_per_seq: int):
        """(block_tables [S][M] int32, context_lens [S] int32) as CPU tensors."""
        ids = torch.as_tensor(list(seq_ids), dtype=torch.int64)
        tables = torch.empty(len(ids), max_blocks_per_seq, dtype=torch.int32)
        lens = torch.empty(len(ids), dtype=torch.int32)
        _bm_check(self._L.pkv_bm_block_tables(self._h, ids.data_ptr(), len(ids),
                                              max_blocks_per_seq, tables.data_ptr(),
                                              lens.data_ptr()))
        return tables, lens

    def prepared_step(self, seq_ids, num_tokens, max_blocks_per_seq: int) -> "PreparedBmStep":
        """A decode step's two calls (append_batch, block_tables) for a fixed batch,
        with their argument and output buffers made once (see PreparedBmStep)."""
        return PreparedBmStep(self, seq_ids, num_tokens, max_blocks_per_seq)

    def table(self, seq: int) -> list:
        width = max(1, self.stats().num_blocks)
        while True:
            try:
                t, _ = self.block_tables([seq], width)
            except PkvError:
                if width >= 1 << 24:
                    raise
                width *= 4      # a prefix can repeat a block, so a table may exceed the pool
                continue
            return [int(b) for b in t[0].tolist() if b >= 0]

    def stats(self) -> BmStats:
        st = BmStats()
        _bm_check(self._L.pkv_bm_stats_get(self._h, ctypes.byref(st)))
        return st

    def refcount(self, block: int) -> int:
        return int(self._L.pkv_bm_refcount(self._h, block))

    def num_free(self) -> int:
        return int(self.stats().free_blocks)


def simulate_admission(num_blocks: int, block_size: int, context_lens, reserve_tokens: int = 0):
    """(admitted, utilisation) of requests admitted in order into a pool."""
    L = _bm_lib()
    cl = torch.as_tensor(list(context_lens), dtype=torch.int32)
    adm = ctypes.c_int32(0)
    u = ctypes.c_double(0.0)
    _bm_check(L.pkv_bm_simulate_admission(num_blocks, block_size, cl.data_ptr(), len(cl),
                                          reserve_tokens, ctypes.byref(adm), ctypes.byref(u)))
    return int(adm.value), float(u.value)


# ------------------------------------------------------------------ flat spans
class FlatInfo(ctypes.Structure):
    _fields_ = [("k_base", ctypes.c_void_p), ("slot_stride", ctypes.c_size_t),
                ("v_offset", ctypes.c_size_t), ("granularity", ctypes.c_size_t),
                ("committed_bytes", ctypes.c_size_t), ("committed_tokens", ctypes.c_void_p)]


def _flat_lib():
    L = lib()
    if not getattr(L, "_flat_ready", False):
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.pkv_flat_create.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.pkv_flat_create.restype = i32
        L.pkv_flat_destroy.argtypes = [vp]
        L.pkv_flat_destroy.restype = None
        L.pkv_flat_reserve.argtypes = [vp, i32, i32]
        L.pkv_flat_reserve.restype = i32
        L.pkv_flat_release.argtypes = [vp, i32]
        L.pkv_flat_release.restype = i32
        L.pkv_flat_get_info.argtypes = [vp, ctypes.POINTER(FlatInfo)]
        L.pkv_flat_get_info.restype = i32
        L.pkv_flat_append.argtypes = [vp, vp, vp, vp, vp, i32, vp]
        L.pkv_flat_append.restype = i32
        L.pkv_flat_decode_workspace_bytes.argtypes = [vp, i32, i32]
        L.pkv_flat_decode_workspace_bytes.restype = sz
        L.pkv_decode_attention_flat.argtypes = [vp, vp, i32, i32, vp, vp, ctypes.c_float, vp, i32,
                                                vp, sz, vp, ctypes.POINTER(DecodeOptions)]
        L.pkv_decode_attention_flat.restype = i32
        L._flat_ready = True
    return L


class FlatCache:
    """A KV cache kept contiguous in virtual memory (libpkv's pkv_flat_* calls):
    num_slots sequence slots of capacity tokens, physical chunks mapped as
    slots grow."""

    def __init__(self, num_slots: int, capacity: int, num_kv_heads: int, head_dim: int,
                 dtype: torch.dtype):
        L = _flat_lib()
        h = ctypes.c_void_p()
        _check(L.pkv_flat_create(num_slots, capacity, num_kv_heads, head_dim, DTYPE_CODE[dtype],
                                 ctypes.byref(h)))
        self._h, self._L = h, L
        self.num_slots, self.capacity = num_slots, capacity
        self.num_kv_heads, self.head_dim, self.dtype = num_kv_heads, head_dim, dtype

    def close(self):
        if getattr(self, "_h", None):
            self._L.pkv_flat_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def reserve(self, slot: int, tokens: int) -> None:
        _check(self._L.pkv_flat_reserve(self._h, slot, tokens))

    def release(self, slot: int) -> None:
        _check(self._L.pkv_flat_release(self._h, slot))

    def info(self) -> FlatInfo:
        inf = FlatInfo()
        _check(self._L.pkv_flat_get_info(self._h, ctypes.byref(inf)))
        return inf

    def append(self, k_new, v_new, slots, positions, stream=None) -> None:
        """k_new/v_new [N][Hk][D] (device); slots/positions int32 [N] (device)."""
        k_new, v_new = k_new.contiguous(), v_new.contiguous()
        sl, pos = slots.contiguous(), positions.contiguous()
        assert sl.dtype == torch.int32 and pos.dtype == torch.int32 and k_new.dtype == self.dtype
        _check(self._L.pkv_flat_append(self._h, _ptr(k_new), _ptr(v_new), _ptr(sl), _ptr(pos),
                                       sl.numel(), _stream(stream)))

    def workspace(self, num_q_heads: int, num_ctas: int = 0) -> torch.Tensor:
        n = int(self._L.pkv_flat_decode_workspace_bytes(self._h, num_q_heads, num_ctas))
        if n == 0:
            raise PkvError(-1, "workspace size query failed")
        return torch.zeros(n, dtype=torch.uint8, device="cuda")

    def decode_attention(self, q, slots, context_lens, scale: float,
                         out: Optional[torch.Tensor] = None,
                         out_dtype: Optional[torch.dtype] = None,
                         workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                         timing_events: Optional[Sequence] = None, stream=None,
                         tables_ready: bool = False, pending_tail: int = 0) -> torch.Tensor:
        S, Hq, D = q.shape
        q = q.contiguous()
        sl, cl = slots.contiguous(), context_lens.contiguous()
        assert sl.dtype == torch.int32 and cl.dtype == torch.int32 and q.dtype == self.dtype
        if out is None:
            out = torch.empty(S, Hq, D, dtype=out_dtype or q.dtype, device=q.device)
        if workspace is None:
            workspace = self.workspace(Hq, num_ctas)
        opts = DecodeOptions()
        opts.num_ctas = num_ctas
        opts.tables_ready = int(tables_ready)
        opts.pending_tail = int(pending_tail)
        if timing_events is not None:
            for i, ev in enumerate(timing_events):
                opts.timing_events[i] = None if ev is None else ev.cuda_event
        _check(self._L.pkv_decode_attention_flat(
            self._h, _ptr(q), S, Hq, _ptr(sl), _ptr(cl), float(scale), _ptr(out),
            DTYPE_CODE[out.dtype], _ptr(workspace), workspace.numel(), _stream(stream),
            ctypes.byref(opts)))
        return out


# ------------------------------------------------------------------ prefix-aware decode
class _Groups:
    """Host arrays of a prefix-group description, kept alive with the struct."""

    def __init__(self, group_of_seq, group_prefix_blocks):
        self.gos = torch.as_tensor(list(group_of_seq), dtype=torch.int32).contiguous()
        self.gpb = torch.as_tensor(list(group_prefix_blocks), dtype=torch.int32).contiguous()
        self.st = PrefixGroups(len(self.gpb), self.gos.data_ptr() if len(self.gos) else None,
                               self.gpb.data_ptr() if len(self.gpb) else None)


def prefix_workspace_bytes(k_pool, num_seqs, num_q_heads, max_blocks_per_seq, group_of_seq,
                           group_prefix_blocks, num_ctas: int = 0) -> int:
    g = _Groups(group_of_seq, group_prefix_blocks)
    desc = cache_desc(k_pool)
    return int(lib().pkv_decode_prefix_workspace_bytes(ctypes.byref(desc), num_seqs, num_q_heads,
                                                       max_blocks_per_seq, ctypes.byref(g.st),
                                                       num_ctas))


def decode_attention_prefix(q, k_pool, v_pool, block_tables, context_lens, scale: float,
                            group_of_seq, group_prefix_blocks,
                            out: Optional[torch.Tensor] = None,
                            out_dtype: Optional[torch.dtype] = None,
                            workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                            stream=None, lse_out: Optional[torch.Tensor] = None,
                            tables_ready: bool = False, consumer: int = 0) -> torch.Tensor:
    """Decode where the sequences of each group share their first
    group_prefix_blocks[g] table entries (group_of_seq[s] = g, or -1)."""
    return PreparedDecodePrefix(q, k_pool, v_pool, block_tables, context_lens, scale,
                                group_of_seq, group_prefix_blocks, out=out, out_dtype=out_dtype,
                                workspace=workspace, num_ctas=num_ctas, lse_out=lse_out,
                                tables_ready=tables_ready, consumer=consumer)(stream)


class PreparedDecodePrefix:
    """A pkv_decode_attention_prefix call whose arguments (and group arrays)
    are marshalled once; each call passes the stream (see PreparedDecode)."""

    def __init__(self, q, k_pool, v_pool, block_tables, context_lens, scale: float,
                 group_of_seq, group_prefix_blocks, out: Optional[torch.Tensor] = None,
                 out_dtype: Optional[torch.dtype] = None,
                 workspace: Optional[torch.Tensor] = None, num_ctas: int = 0,
                 lse_out: Optional[torch.Tensor] = None, tables_ready: bool = False,
                 consumer: int = 0):
        self._desc = _pools(k_pool, v_pool)
        S, Hq, D = q.shape
        q = q.contiguous()
        bt, cl = block_tables.contiguous(), context_lens.contiguous()
        assert bt.dtype == torch.int32 and cl.dtype == torch.int32 and q.dtype == k_pool.dtype
        self._g = _Groups(group_of_seq, group_prefix_blocks)
        if out is None:
            out = torch.empty(S, Hq, D, dtype=out_dtype or q.dtype, device=q.device)
        if workspace is None:
            n = prefix_workspace_bytes(k_pool, S, Hq, bt.shape[1], group_of_seq,
                                       group_prefix_blocks, num_ctas)
            if n == 0:
                raise PkvError(-1, lib().pkv_last_error_message().decode())
            workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
        self._opts = DecodeOptions()
        self._opts.num_ctas = num_ctas
        self._opts.consumer = consumer
        self._opts.tables_ready = int(tables_ready)
        if lse_out is not None:
            assert lse_out.dtype == torch.float32 and lse_out.shape == (S, Hq) and lse_out.is_contiguous()
            self._opts.lse_out = lse_out.data_ptr()
        self._keep = (q, k_pool, v_pool, bt, cl, out, workspace, lse_out)
        self._args = (ctypes.byref(self._desc), _ptr(q), S, Hq, _ptr(k_pool), _ptr(v_pool),
                      _ptr(bt), bt.shape[1], _ptr(cl), float(scale), ctypes.byref(self._g.st),
                      _ptr(out), DTYPE_CODE[out.dtype], _ptr(workspace), workspace.numel())
        self._fn = lib().pkv_decode_attention_prefix
        self.out = out
        self.workspace = workspace

    def __call__(self, stream=None, timing_events: Optional[Sequence] = None) -> torch.Tensor:
        opts = self._opts
        for i in range(2):
            ev = timing_events[i] if timing_events is not None else None
            opts.timing_events[i] = None if ev is None else ev.cuda_event
        _check(self._fn(*self._args, _stream(stream), ctypes.byref(opts)))
        return self.out
