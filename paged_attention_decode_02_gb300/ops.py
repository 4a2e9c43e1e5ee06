"""ctypes binding of libpa_decode.so (see include/pa_decode.h).

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch supplies device memory and the
current stream); the library allocates nothing.  If the shared library is missing
the calls raise -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_decode.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = 0, -1, -2, -3, -4
PA_KV_BF16, PA_KV_FP8_E4M3, PA_KV_MXFP4 = 0, 1, 2
PA_SCALE_NONE, PA_SCALE_PER_TENSOR, PA_SCALE_PER_TOKEN, PA_SCALE_E8M0_32 = 0, 1, 2, 3
PA_Q_BF16, PA_Q_FP8_E4M3, PA_Q_BF16_TO_E4M3 = 0, 1, 2
PA_DEVICE_WAIT_TIMEOUT, PA_DEVICE_CONTEXT_CLAMPED = 1, 2
PA_KERNEL_DEFAULT, PA_KERNEL_MMA, PA_KERNEL_TCGEN05 = 0, 1, 2
_KERNELS = {None: PA_KERNEL_DEFAULT, "default": PA_KERNEL_DEFAULT, "mma": PA_KERNEL_MMA,
            "tc": PA_KERNEL_TCGEN05, "tcgen05": PA_KERNEL_TCGEN05}

EXPORTED = ["pa_decode_abi_version", "pa_decode_workspace_size", "pa_decode_validate",
            "pa_decode_plan", "pa_decode", "pa_decode_reduce", "pa_decode_run",
            "pa_decode_read_status", "pa_status_string", "pa_decode_run_static",
            "pa_decode_read_status_static", "pa_mxfp4_kv_write"]
STATIC_WORKSPACE_BYTES = 16 << 20


class PaDecodeArgs(ctypes.Structure):
    """Mirror of ``pa_decode_args``."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("qlen", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("kv_scale", ctypes.c_int32), ("q_dtype", ctypes.c_int32),
        ("q_scale_per_row", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
        ("max_partitions", ctypes.c_int32), ("task_budget", ctypes.c_int32),
        ("merge_in_decode", ctypes.c_int32),
        ("query", ctypes.c_void_p), ("q_stride_token", ctypes.c_int64),
        ("q_stride_head", ctypes.c_int64), ("q_scale", ctypes.c_void_p),
        ("key_cache", ctypes.c_void_p), ("value_cache", ctypes.c_void_p),
        ("kv_stride_block", ctypes.c_int64), ("kv_stride_head", ctypes.c_int64),
        ("kv_stride_token", ctypes.c_int64), ("key_scale", ctypes.c_void_p),
        ("value_scale", ctypes.c_void_p), ("scale_stride_block", ctypes.c_int64),
        ("scale_stride_head", ctypes.c_int64), ("block_tables", ctypes.c_void_p),
        ("bt_stride", ctypes.c_int64), ("context_lens", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_stride_token", ctypes.c_int64),
        ("out_stride_head", ctypes.c_int64), ("causal", ctypes.c_int32),
        ("sliding_window", ctypes.c_int32), ("trans_v", ctypes.c_int32),
        ("sinks", ctypes.c_void_p), ("kernel", ctypes.c_int32),
    ]


class PaDecodeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Open libpa_decode.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with "
                               "paged_attention_decode_02_gb300.build.build()")
        L = ctypes.CDLL(p)
        A = ctypes.POINTER(PaDecodeArgs)
        L.pa_decode_abi_version.restype = ctypes.c_int32
        L.pa_decode_workspace_size.argtypes = [A]
        L.pa_decode_workspace_size.restype = ctypes.c_size_t
        L.pa_decode_validate.argtypes = [A]
        L.pa_decode_validate.restype = ctypes.c_int32
        for name in ("pa_decode_plan", "pa_decode", "pa_decode_reduce", "pa_decode_run"):
            f = getattr(L, name)
            f.argtypes = [A, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
            f.restype = ctypes.c_int32
        L.pa_decode_run_static.argtypes = [A, ctypes.c_void_p]
        L.pa_decode_run_static.restype = ctypes.c_int32
        L.pa_decode_read_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.pa_decode_read_status.restype = ctypes.c_int32
        L.pa_decode_read_status_static.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        L.pa_decode_read_status_static.restype = ctypes.c_int32
        L.pa_status_string.argtypes = [ctypes.c_int32]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_mxfp4_kv_write.argtypes = [ctypes.POINTER(Mxfp4WriteArgs), ctypes.c_void_p]
        L.pa_mxfp4_kv_write.restype = ctypes.c_int32
        if path is None:
            _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return load_library().pa_status_string(status).decode()
    except Exception:  # library not built: still give a readable message
        return {0: "ok", -1: "invalid argument", -2: "unsupported combination",
                -3: "workspace", -4: "CUDA error"}.get(status, "unknown status")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def call_device(tensors, stream=None) -> torch.device:
    """The one CUDA device a call's tensors live on; raises ValueError when they are spread
    over several devices, are not CUDA tensors, or when ``stream`` (a torch stream) belongs to
    another device.  The library launches on the current device and stream, so callers make
    this device current for the call."""
    devs = {t.device for t in tensors if t is not None}
    if len(devs) != 1 or next(iter(devs)).type != "cuda":
        raise ValueError(f"every tensor must be on one CUDA device, got {devs}")
    dev = next(iter(devs))
    sdev = getattr(stream, "device", None)
    if sdev is not None and torch.device(sdev) != dev:
        raise ValueError(f"stream is on {sdev}, the tensors on {dev}")
    return dev


def _check_tensor(t: torch.Tensor, name: str, dtypes, *, contiguous_last=True):
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected one of {[str(d) for d in dtypes]}")
    if contiguous_last and t.dim() > 0 and t.stride(-1) != 1:
        raise ValueError(f"{name}: the last axis must be contiguous (stride 1)")


def make_args(query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor, out: torch.Tensor, *,
              key_scale: Optional[torch.Tensor] = None, value_scale: Optional[torch.Tensor] = None,
              q_scale: Optional[torch.Tensor] = None, softmax_scale: Optional[float] = None,
              max_partitions: int = 0, task_budget: int = 0,
              merge_in_decode: bool = False, causal: bool = False,
              q_quant: bool = False, sliding_window: int = 0,
              trans_v: bool = False, sinks: Optional[torch.Tensor] = None,
              kernel=None) -> PaDecodeArgs:
    """Describe one decode call.

    query / out: [B, qlen, Hq, D] (or [B*qlen, Hq, D]); query bf16 or e4m3
    (torch.float8_e4m3fn or uint8 bytes with ``q_scale``); out bf16.
    key_cache / value_cache: [NB, Hkv, S, D] bf16, [NB, Hkv, S, D] e4m3 bytes
    (uint8 / float8_e4m3fn) with fp32 scales [1] (per tensor) or [NB, Hkv, S]
    (per token), or [NB, Hkv, S, D/2] uint8 MXFP4 with uint8 e8m0 scales
    [NB, Hkv, S, D/32].  block_tables int32 [B, W]; context_lens int32 [B].
    causal: query position i sees tokens < L - qlen + 1 + i.  sliding_window W > 0: query
    position i sees only tokens > L - qlen + i - W.  trans_v: value_cache is [NB, Hkv, D, S]
    (e4m3 bytes, per-tensor scale), with the key cache's block and head strides.
    sinks: fp32 [Hq], one softmax logit per query head with a zero value, or None.
    kernel: None / "default" (the library's choice), "mma" (the mma.sync tile kernel) or
    "tc" (the tcgen05 kernel where it covers the shape).
    Malformed tensors (wrong dtype, shape, batch or layout) raise ValueError here, before
    any pointer reaches the library.
    """
    _check_tensor(query, "query", (torch.bfloat16, torch.float8_e4m3fn, torch.uint8))
    _check_tensor(out, "out", (torch.bfloat16,))
    if tuple(out.shape) != tuple(query.shape):
        raise ValueError(f"out {tuple(out.shape)} must have the query's shape {tuple(query.shape)}")
    if query.dim() not in (3, 4):
        raise ValueError("query: [B, qlen, Hq, D] or [B*qlen, Hq, D]")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name}: contiguous int32 expected, got {t.dtype}")
    if block_tables.dim() != 2 or context_lens.dim() != 1:
        raise ValueError("block_tables [B, W] and context_lens [B]")
    B_ = block_tables.shape[0]
    if context_lens.shape[0] != B_:
        raise ValueError(f"context_lens has {context_lens.shape[0]} entries for {B_} sequences")
    if query.dim() == 4 and query.shape[0] != B_:
        raise ValueError(f"query batch {query.shape[0]} != block_tables batch {B_}")
    if query.dim() == 3 and (B_ == 0 or query.shape[0] % B_):
        raise ValueError("query rows must be batch x qlen")
    if key_cache.dtype != value_cache.dtype:
        raise ValueError(f"key cache {key_cache.dtype} and value cache {value_cache.dtype} differ")
    _check_tensor(key_cache, "key_cache", (torch.bfloat16, torch.uint8, torch.float8_e4m3fn))
    if key_cache.dim() != 4 or value_cache.dim() != 4:
        raise ValueError("caches: 4-D [NB, Hkv, S, row]")
    if kernel not in _KERNELS:
        raise ValueError(f"kernel: one of {sorted(k for k in _KERNELS if k)} or None")
    D = query.shape[-1]
    Hq = query.shape[-2]
    if query.dim() == 4:
        B, qlen = query.shape[0], query.shape[1]
        q_st, q_sh = query.stride(1), query.stride(2)
        if query.stride(0) != qlen * q_st:
            raise ValueError("query sequence and position axes must be fused-contiguous")
    else:
        B, qlen = block_tables.shape[0], query.shape[0] // max(1, block_tables.shape[0])
        q_st, q_sh = query.stride(0), query.stride(1)
    o_st = out.stride(-3) if out.dim() == 3 else out.stride(1)
    o_sh = out.stride(-2)
    NB, Hkv, S = key_cache.shape[0], key_cache.shape[1], key_cache.shape[2]
    a = PaDecodeArgs()
    a.batch, a.qlen, a.num_q_heads, a.num_kv_heads = B, qlen, Hq, Hkv
    a.head_dim, a.page_size, a.num_blocks = D, S, NB
    a.max_blocks_per_seq = block_tables.shape[1]
    if key_cache.dtype == torch.bfloat16:
        a.kv_dtype, a.kv_scale = PA_KV_BF16, PA_SCALE_NONE
    elif key_cache.shape[-1] == D:
        a.kv_dtype = PA_KV_FP8_E4M3
        if key_scale is None or value_scale is None:
            raise ValueError("fp8 KV needs key_scale and value_scale")
        for t, name in ((key_scale, "key_scale"), (value_scale, "value_scale")):
            if t.dtype != torch.float32:
                raise ValueError(f"{name}: fp32 expected for an e4m3 cache, got {t.dtype}")
        if key_scale.numel() != value_scale.numel():
            raise ValueError("key_scale and value_scale must have the same shape")
        a.kv_scale = PA_SCALE_PER_TENSOR if key_scale.numel() == 1 else PA_SCALE_PER_TOKEN
        if a.kv_scale == PA_SCALE_PER_TOKEN and (tuple(key_scale.shape) != (NB, Hkv, S)
                                                 or key_scale.stride(-1) != 1):
            raise ValueError(f"per-token scales: fp32 [NB, Hkv, S] = {(NB, Hkv, S)}, token axis dense")
    elif key_cache.shape[-1] * 2 == D:
        a.kv_dtype, a.kv_scale = PA_KV_MXFP4, PA_SCALE_E8M0_32
        if key_scale is None or value_scale is None:
            raise ValueError("MXFP4 KV needs e8m0 key_scale and value_scale")
        for t, name in ((key_scale, "key_scale"), (value_scale, "value_scale")):
            if t.dtype != torch.uint8 or tuple(t.shape) != (NB, Hkv, S, D // 32) \
                    or t.stride(-1) != 1 or t.stride(-2) != D // 32:
                raise ValueError(f"{name}: uint8 e8m0 [NB, Hkv, S, D/32] = {(NB, Hkv, S, D // 32)}, "
                                 "token rows dense")
    else:
        raise ValueError(f"cannot infer the KV format from {tuple(key_cache.shape)} and D={D}")
    if query.dtype == torch.bfloat16:
        a.q_dtype = PA_Q_BF16_TO_E4M3 if q_quant else PA_Q_BF16
    else:
        a.q_dtype = PA_Q_FP8_E4M3
        if q_scale is None or q_scale.dtype != torch.float32:
            raise ValueError("an e4m3 query needs an fp32 q_scale ([1] or [B, qlen, Hq])")
    if a.kv_dtype == PA_KV_BF16 and (key_scale is not None or value_scale is not None):
        raise ValueError("bf16 KV takes no scales")
    a.q_scale_per_row = int(q_scale is not None and q_scale.numel() > 1)
    a.softmax_scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(D)
    a.max_partitions, a.task_budget = int(max_partitions), int(task_budget)
    a.merge_in_decode = int(bool(merge_in_decode))
    a.causal = int(bool(causal))
    a.sliding_window = int(sliding_window)
    a.trans_v = int(bool(trans_v))
    if sinks is not None and (sinks.dtype != torch.float32 or sinks.numel() != Hq):
        raise ValueError("sinks: fp32, one per query head")
    a.sinks = _ptr(sinks)
    a.kernel = _KERNELS[kernel]
    a.query, a.q_stride_token, a.q_stride_head = _ptr(query), q_st, q_sh
    a.q_scale = _ptr(q_scale)
    es = key_cache.element_size()
    a.key_cache, a.value_cache = _ptr(key_cache), _ptr(value_cache)
    if trans_v:
        if value_cache.stride()[:2] != key_cache.stride()[:2] or value_cache.stride(-1) != 1 \
                or value_cache.stride(-2) != S:
            raise ValueError("a transposed value cache is [NB, Hkv, D, S], dense pages, with "
                             "the key cache's block and head strides")
    elif value_cache.stride() != key_cache.stride():
        raise ValueError("key and value caches must share strides")
    a.kv_stride_block = key_cache.stride(0) * es
    a.kv_stride_head = key_cache.stride(1) * es
    a.kv_stride_token = key_cache.stride(2) * es
    a.key_scale, a.value_scale = _ptr(key_scale), _ptr(value_scale)
    if a.kv_scale in (PA_SCALE_PER_TOKEN, PA_SCALE_E8M0_32):
        ses = key_scale.element_size()
        a.scale_stride_block = key_scale.stride(0) * ses
        a.scale_stride_head = key_scale.stride(1) * ses
    a.block_tables, a.bt_stride = _ptr(block_tables), block_tables.stride(0)
    a.context_lens = _ptr(context_lens)
    a.out, a.out_stride_token, a.out_stride_head = _ptr(out), o_st, o_sh
    return a


def _check(status: int, what: str):
    if status != PA_OK:
        raise PaDecodeError(status, what)


def pa_decode_validate(args: PaDecodeArgs) -> int:
    return load_library().pa_decode_validate(ctypes.byref(args))


def pa_decode_workspace_size(args: PaDecodeArgs) -> int:
    n = load_library().pa_decode_workspace_size(ctypes.byref(args))
    if n == 0:
        _check(pa_decode_validate(args) or PA_ERR_CUDA, "pa_decode_workspace_size")
    return n


def alloc_workspace(args: PaDecodeArgs, device=None) -> torch.Tensor:
    """Caller-side workspace allocation (torch memory, 256-byte aligned)."""
    n = pa_decode_workspace_size(args)
    return torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")


def _ws(workspace: torch.Tensor):
    base = workspace.data_ptr()
    off = (-base) % 256
    return base + off, workspace.numel() - off


def pa_decode_plan(args: PaDecodeArgs, workspace: torch.Tensor, stream=None):
    p, n = _ws(workspace)
    _check(load_library().pa_decode_plan(ctypes.byref(args), p, n, _stream_handle(stream)),
           "pa_decode_plan")


def pa_decode(args: PaDecodeArgs, workspace: torch.Tensor, stream=None):
    p, n = _ws(workspace)
    _check(load_library().pa_decode(ctypes.byref(args), p, n, _stream_handle(stream)), "pa_decode")


def pa_decode_reduce(args: PaDecodeArgs, workspace: torch.Tensor, stream=None):
    p, n = _ws(workspace)
    _check(load_library().pa_decode_reduce(ctypes.byref(args), p, n, _stream_handle(stream)),
           "pa_decode_reduce")


def pa_decode_run(args: PaDecodeArgs, workspace: torch.Tensor, stream=None):
    p, n = _ws(workspace)
    _check(load_library().pa_decode_run(ctypes.byref(args), p, n, _stream_handle(stream)),
           "pa_decode_run")


def pa_decode_run_static(args: PaDecodeArgs, stream=None):
    """plan + decode + reduce with the library's fixed device workspace, for callers that
    cannot allocate device memory (see include/pa_decode.h).  Nothing is allocated."""
    status = load_library().pa_decode_run_static(ctypes.byref(args), _stream_handle(stream))
    if status == PA_ERR_WORKSPACE:
        raise PaDecodeError(status, f"pa_decode_run_static: the problem needs "
                                    f"{pa_decode_workspace_size(args)} bytes of workspace, more "
                                    f"than the fixed {STATIC_WORKSPACE_BYTES}")
    _check(status, "pa_decode_run_static")


def pa_decode_read_status_static(stream=None) -> int:
    """Device status word of the last pa_decode_run_static call on the current device;
    synchronises the stream."""
    host = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    _check(load_library().pa_decode_read_status_static(host.data_ptr(), _stream_handle(stream)),
           "pa_decode_read_status_static")
    (stream or torch.cuda.current_stream()).synchronize()
    return int(host.item())


def pa_decode_read_status(workspace: torch.Tensor, stream=None) -> int:
    """Device status word (PA_DEVICE_* bits); synchronises the stream."""
    host = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    p, _ = _ws(workspace)
    _check(load_library().pa_decode_read_status(p, host.data_ptr(), _stream_handle(stream)),
           "pa_decode_read_status")
    (stream or torch.cuda.current_stream()).synchronize()
    return int(host.item())


def paged_attention_decode(query: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                           key_scale: Optional[torch.Tensor] = None,
                           value_scale: Optional[torch.Tensor] = None,
                           q_scale: Optional[torch.Tensor] = None,
                           softmax_scale: Optional[float] = None, max_partitions: int = 0,
                           causal: bool = False, sliding_window: int = 0, trans_v: bool = False,
                           sinks: Optional[torch.Tensor] = None, q_quant: bool = False,
                           kernel=None, workspace: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """One decode call on tensors: plan + decode + reduce on ``stream`` (default: the
    current stream of the tensors' device), returning ``out`` (bf16, the query's shape;
    allocated when not given).  The arguments are those of make_args; ``workspace`` (from
    alloc_workspace) is allocated per call when not given.  Every tensor must be on one
    CUDA device, which is made current for the call, and an explicit stream must belong
    to it (ValueError otherwise); a refused call raises PaDecodeError.  Nothing here
    computes: the library does the work."""
    dev = call_device([query, key_cache, value_cache, block_tables, context_lens, out,
                       key_scale, value_scale, q_scale, sinks, workspace], stream)
    with torch.cuda.device(dev):
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        if query.dtype == torch.uint8:
            query = query.view(torch.float8_e4m3fn)
        if out is None:
            out = torch.empty(query.shape, dtype=torch.bfloat16, device=dev)
        args = make_args(query, key_cache, value_cache, block_tables, context_lens, out,
                         key_scale=key_scale, value_scale=value_scale, q_scale=q_scale,
                         softmax_scale=softmax_scale, max_partitions=max_partitions,
                         causal=causal, q_quant=q_quant, sliding_window=sliding_window,
                         trans_v=trans_v, sinks=sinks, kernel=kernel)
        if workspace is None:
            workspace = alloc_workspace(args, dev)
        pa_decode_run(args, workspace, stream)
    return out


def decode(problem: dict, out: Optional[torch.Tensor] = None, *, max_partitions: int = 0,
           task_budget: int = 0, workspace: Optional[torch.Tensor] = None,
           merge_in_decode: bool = False, kernel=None):
    """plan + decode + reduce on a synthetic-workload dict (device tensors)."""
    case = problem["case"]
    q = problem["query"]
    if q.dtype == torch.uint8:
        q = q.view(torch.float8_e4m3fn)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    args = make_args(q, problem["key_cache"], problem["value_cache"], problem["block_tables"],
                     problem["context_lens"], out, key_scale=problem["key_scale"],
                     value_scale=problem["value_scale"], q_scale=problem["q_scale"],
                     softmax_scale=case.scale_qk(), max_partitions=max_partitions,
                     task_budget=task_budget, merge_in_decode=merge_in_decode,
                     causal=getattr(case, "causal", False), q_quant=getattr(case, "q_quant", False),
                     sliding_window=getattr(case, "window", 0),
                     trans_v=getattr(case, "trans_v", False), sinks=problem.get("sinks"),
                     kernel=kernel)
    if workspace is None:
        workspace = alloc_workspace(args, q.device)
    pa_decode_run(args, workspace)
    return out, args, workspace


class Mxfp4WriteArgs(ctypes.Structure):
    """Mirror of ``pa_mxfp4_write_args`` (include/pa_kv_write.h)."""
    _fields_ = [
        ("num_tokens", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32), ("key", ctypes.c_void_p), ("value", ctypes.c_void_p),
        ("src_stride_token", ctypes.c_int64), ("src_stride_head", ctypes.c_int64),
        ("slot_mapping", ctypes.c_void_p), ("key_cache", ctypes.c_void_p),
        ("value_cache", ctypes.c_void_p), ("cache_stride_block", ctypes.c_int64),
        ("cache_stride_head", ctypes.c_int64), ("key_scale", ctypes.c_void_p),
        ("value_scale", ctypes.c_void_p), ("scale_stride_block", ctypes.c_int64),
        ("scale_stride_head", ctypes.c_int64),
    ]


def mxfp4_write_args(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
                     key_cache: torch.Tensor, value_cache: torch.Tensor,
                     key_scale: torch.Tensor, value_scale: torch.Tensor) -> Mxfp4WriteArgs:
    """key / value bf16 [T, Hkv, D]; slot_mapping int64 [T]; caches uint8 [NB, Hkv, S, D/2]
    and e8m0 scales uint8 [NB, Hkv, S, D/32] (token rows dense)."""
    if key.stride() != value.stride() or key.dtype != torch.bfloat16 or value.dtype != torch.bfloat16:
        raise ValueError("key and value: bf16 [T, Hkv, D] with the same strides")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if key_cache.stride() != value_cache.stride() or key_scale.stride() != value_scale.stride():
        raise ValueError("key and value caches (and scale caches) must share strides")
    a = Mxfp4WriteArgs()
    a.num_tokens, a.num_kv_heads, a.head_dim = key.shape[0], key.shape[1], key.shape[2]
    a.num_blocks, a.page_size = key_cache.shape[0], key_cache.shape[2]
    a.key, a.value = _ptr(key), _ptr(value)
    a.src_stride_token, a.src_stride_head = key.stride(0), key.stride(1)
    a.slot_mapping = _ptr(slot_mapping)
    a.key_cache, a.value_cache = _ptr(key_cache), _ptr(value_cache)
    a.cache_stride_block, a.cache_stride_head = key_cache.stride(0), key_cache.stride(1)
    a.key_scale, a.value_scale = _ptr(key_scale), _ptr(value_scale)
    a.scale_stride_block, a.scale_stride_head = key_scale.stride(0), key_scale.stride(1)
    return a


def mxfp4_kv_write(args: Mxfp4WriteArgs, stream=None):
    """Quantise and write the rows described by ``args`` (see include/pa_kv_write.h)."""
    _check(load_library().pa_mxfp4_kv_write(ctypes.byref(args), _stream_handle(stream)),
           "pa_mxfp4_kv_write")
