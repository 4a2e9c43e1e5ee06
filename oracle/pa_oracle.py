"""ctypes binding of the fp64 CPU oracle for paged-attention decode.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The library is plain C
(``pa_oracle.c``), compiled here with gcc; it shares no code with the CUDA path
and never imports it.

Inputs are the same stored bytes the GPU path reads (dense, contiguous numpy
arrays or CPU torch tensors); the result is float64 ``[B, qlen, Hq, D]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpa_oracle.so")

KV_BF16, KV_E4M3, KV_MXFP4 = 0, 1, 2
SCALE_NONE, SCALE_TENSOR, SCALE_TOKEN, SCALE_E8M0 = 0, 1, 2, 3
Q_BF16, Q_E4M3, Q_BF16_TO_E4M3 = 0, 1, 2


class OrcArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("qlen", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("kv_format", ctypes.c_int32),
        ("scale_kind", ctypes.c_int32),
        ("q_format", ctypes.c_int32),
        ("q_scale_per_row", ctypes.c_int32),
        ("softmax_scale", ctypes.c_double),
        ("query", ctypes.c_void_p),
        ("q_scale", ctypes.c_void_p),
        ("key_cache", ctypes.c_void_p),
        ("value_cache", ctypes.c_void_p),
        ("key_scale", ctypes.c_void_p),
        ("value_scale", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p),
        ("context_lens", ctypes.c_void_p),
        ("causal", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("trans_v", ctypes.c_int32),
        ("sinks", ctypes.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.orc_pa_decode.argtypes = [ctypes.POINTER(OrcArgs), ctypes.c_void_p, ctypes.c_int]
            L.orc_pa_decode.restype = ctypes.c_int
            L.orc_pa_decode_range.argtypes = [ctypes.POINTER(OrcArgs), ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p]
            L.orc_pa_decode_range.restype = ctypes.c_int
            for name in ("orc_e4m3", "orc_e2m1", "orc_e8m0"):
                getattr(L, name).argtypes = [ctypes.c_uint8]
                getattr(L, name).restype = ctypes.c_double
            L.orc_bf16.argtypes = [ctypes.c_uint16]
            L.orc_bf16.restype = ctypes.c_double
            L.orc_e4m3_round.argtypes = [ctypes.c_float]
            L.orc_e4m3_round.restype = ctypes.c_double
            L.orc_max_threads.restype = ctypes.c_int
            L.orc_mxfp4_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_void_p]
            L.orc_mxfp4_quantize.restype = ctypes.c_int
            _lib = L
        return _lib


def _np(x, dtype=None):
    """Contiguous numpy view of a CPU tensor or array (raw bytes preserved)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: reinterpret as bytes, then as dtype
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype in (torch.bfloat16, torch.float8_e4m3fn, torch.float8_e8m0fnu,
                       torch.uint8, torch.int8):
            t = t.view(torch.uint8) if t.element_size() == 1 else t.view(torch.int16)
        x = t.numpy()
    x = np.ascontiguousarray(x)
    if dtype is not None:
        x = x.view(dtype) if x.dtype.itemsize == np.dtype(dtype).itemsize else x.astype(dtype)
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data


class Problem:
    """Stored bytes of one decode call, in the dense layouts the oracle reads.

    kv_format: KV_BF16 | KV_E4M3 | KV_MXFP4; scale_kind: SCALE_*; q_format: Q_BF16 | Q_E4M3 |
    Q_BF16_TO_E4M3 (bf16 query quantised per head row to e4m3, scale amax / 448).
    query: [B, qlen, Hq, D] (bf16 bits as uint16/int16, or e4m3 bytes);
    key/value: [NB, Hkv, S, row_bytes] bytes (bf16 as 16-bit words);
    key_scale/value_scale: float32 [1] | float32 [NB, Hkv, S] | uint8 [NB, Hkv, S, D/32].
    """

    def __init__(self, *, batch, qlen, num_q_heads, num_kv_heads, head_dim, page_size,
                 num_blocks, kv_format, scale_kind, q_format, softmax_scale, query,
                 key_cache, value_cache, block_tables, context_lens, key_scale=None,
                 value_scale=None, q_scale=None, causal=False, window=0,
                 trans_v=False, sinks=None):
        self.keep = []
        a = OrcArgs()
        a.batch, a.qlen, a.num_q_heads, a.num_kv_heads = batch, qlen, num_q_heads, num_kv_heads
        a.head_dim, a.page_size, a.num_blocks = head_dim, page_size, num_blocks
        bt = _np(block_tables, np.int32)
        cl = _np(context_lens, np.int32)
        a.max_blocks_per_seq = bt.shape[1] if bt.ndim == 2 else 0
        a.kv_format, a.scale_kind, a.q_format = kv_format, scale_kind, q_format
        a.softmax_scale = float(softmax_scale)
        a.causal = int(bool(causal))
        a.window = int(window)
        a.trans_v = int(bool(trans_v))
        sk = _np(sinks, np.float32) if sinks is not None else None
        a.sinks = _ptr(sk)
        self.keep.append(sk)
        q = _np(query)
        kc, vc = _np(key_cache), _np(value_cache)
        ks = _np(key_scale)
        vs = _np(value_scale)
        qs = _np(q_scale, np.float32) if q_scale is not None else None
        if scale_kind in (SCALE_TENSOR, SCALE_TOKEN):
            ks, vs = ks.astype(np.float32, copy=False), vs.astype(np.float32, copy=False)
        a.q_scale_per_row = int(qs is not None and qs.size > 1)
        for name, arr in (("query", q), ("q_scale", qs), ("key_cache", kc),
                          ("value_cache", vc), ("key_scale", ks), ("value_scale", vs),
                          ("block_tables", bt), ("context_lens", cl)):
            setattr(a, name, _ptr(arr))
            self.keep.append(arr)
        self.args = a
        self.shape = (batch, qlen, num_q_heads, head_dim)

    def decode(self, nthreads: int = 0) -> np.ndarray:
        out = np.zeros(self.shape, dtype=np.float64)
        rc = lib().orc_pa_decode(ctypes.byref(self.args), out.ctypes.data, int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle rejected the problem (rc={rc})")
        return out

    def attend_range(self, s: int, hkv: int, t0: int, t1: int):
        a = self.args
        G = a.num_q_heads // a.num_kv_heads
        R = a.qlen * G
        m = np.zeros(R, np.float64)
        l = np.zeros(R, np.float64)
        o = np.zeros((R, a.head_dim), np.float64)
        rc = lib().orc_pa_decode_range(ctypes.byref(a), s, hkv, t0, t1, m.ctypes.data,
                                       l.ctypes.data, o.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle rejected the range (rc={rc})")
        return m, l, o


def decode_e4m3(b: int) -> float:
    return lib().orc_e4m3(b)


def round_e4m3(y: float) -> float:
    """The oracle's nearest-e4m3 rounding (ties to even, saturating at +-448) of float32 y."""
    return lib().orc_e4m3_round(y)


def decode_e2m1(n: int) -> float:
    return lib().orc_e2m1(n)


def decode_e8m0(b: int) -> float:
    return lib().orc_e8m0(b)


def decode_bf16(bits: int) -> float:
    return lib().orc_bf16(bits)


def max_threads() -> int:
    return lib().orc_max_threads()


def mxfp4_quantize(x: np.ndarray):
    """The oracle's MXFP4 conversion of float32 values [..., D] (D a multiple of 32):
    returns (data uint8 [..., D/2], e8m0 scales uint8 [..., D/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    D = x.shape[-1]
    rows = x.reshape(-1, D)
    data = np.zeros((rows.shape[0], D // 2), np.uint8)
    scales = np.zeros((rows.shape[0], D // 32), np.uint8)
    for r in range(rows.shape[0]):
        rc = lib().orc_mxfp4_quantize(rows[r].ctypes.data, D, data[r].ctypes.data,
                                      scales[r].ctypes.data)
        if rc != 0:
            raise ValueError("head_dim must be a multiple of 32")
    return data.reshape(*x.shape[:-1], D // 2), scales.reshape(*x.shape[:-1], D // 32)
