"""The C ABI: the library loads, exports what include/*.h declare, and refuses malformed
or unsupported arguments on the host (no GPU work)."""
import ctypes
import glob
import os
import re

import pytest

from paged_attention_decode_02_gb300 import build, ops

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(INCLUDE, "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declarations_are_exported(lib):
    names = declared_functions()
    assert set(ops.EXPORTED) == set(names), names
    for n in names:
        assert hasattr(lib, n), n
    assert lib.pa_decode_abi_version() == 6


def test_args_struct_layout_matches_header():
    # 16 int32/float fields, then 19 pointers and int64s, then the causal flag and the
    # sliding window, then trans_v (padded), then the sinks pointer, then the kernel choice
    # (padded)
    assert ctypes.sizeof(ops.PaDecodeArgs) == 64 + 23 * 8
    assert ops.PaDecodeArgs.kernel.offset == 64 + 22 * 8
    assert ops.PaDecodeArgs.query.offset == 64
    assert ops.PaDecodeArgs.causal.offset == 64 + 19 * 8
    assert ops.PaDecodeArgs.sliding_window.offset == 64 + 19 * 8 + 4
    assert ops.PaDecodeArgs.trans_v.offset == 64 + 20 * 8
    assert ops.PaDecodeArgs.sinks.offset == 64 + 21 * 8


def _valid_args():
    a = ops.PaDecodeArgs()
    a.batch, a.qlen, a.num_q_heads, a.num_kv_heads = 4, 1, 16, 1
    a.head_dim, a.page_size, a.num_blocks, a.max_blocks_per_seq = 128, 128, 64, 16
    a.kv_dtype, a.kv_scale, a.q_dtype = ops.PA_KV_FP8_E4M3, ops.PA_SCALE_PER_TOKEN, ops.PA_Q_BF16
    a.softmax_scale, a.max_partitions, a.task_budget = 0.0, 0, 152
    fake = 1 << 20  # host-side validation never dereferences pointers
    a.query, a.q_stride_token, a.q_stride_head = fake, 16 * 128, 128
    a.key_cache, a.value_cache = fake, fake * 2
    a.kv_stride_token, a.kv_stride_head = 128, 128 * 128
    a.kv_stride_block = 128 * 128
    a.key_scale, a.value_scale = fake * 3, fake * 4
    a.scale_stride_head, a.scale_stride_block = 128 * 4, 128 * 4
    a.block_tables, a.bt_stride, a.context_lens = fake * 5, 16, fake * 6
    a.out, a.out_stride_token, a.out_stride_head = fake * 7, 16 * 128, 128
    return a


def test_valid_arguments_pass(lib):
    a = _valid_args()
    assert ops.pa_decode_validate(a) == ops.PA_OK
    assert ops.pa_decode_workspace_size(a) > 0
    # head_dim 64 with 64-byte e4m3 rows
    a.head_dim, a.kv_stride_token, a.q_stride_head, a.out_stride_head = 64, 64, 64, 64
    assert ops.pa_decode_validate(a) == ops.PA_OK
    # a transposed value cache with a per-tensor scale
    a.kv_scale, a.trans_v = ops.PA_SCALE_PER_TENSOR, 1
    assert ops.pa_decode_validate(a) == ops.PA_OK


REFUSED = [
    ("head_dim 96", dict(head_dim=96, q_stride_head=96, out_stride_head=96, kv_stride_token=96),
     ops.PA_ERR_UNSUPPORTED),
    ("mxfp4 head_dim 64", dict(kv_dtype=ops.PA_KV_MXFP4, kv_scale=ops.PA_SCALE_E8M0_32,
                               head_dim=64, kv_stride_token=32), ops.PA_ERR_UNSUPPORTED),
    ("page 48", dict(page_size=48), ops.PA_ERR_UNSUPPORTED),
    ("Hq not a multiple of Hkv", dict(num_q_heads=15, num_kv_heads=2), ops.PA_ERR_INVALID_ARG),
    ("qlen 0", dict(qlen=0), ops.PA_ERR_INVALID_ARG),
    ("G*qlen > 64", dict(qlen=5), ops.PA_ERR_UNSUPPORTED),
    ("bf16 with scales", dict(kv_dtype=ops.PA_KV_BF16), ops.PA_ERR_UNSUPPORTED),
    ("fp8 with e8m0", dict(kv_scale=ops.PA_SCALE_E8M0_32), ops.PA_ERR_UNSUPPORTED),
    ("mxfp4 qlen 2", dict(kv_dtype=ops.PA_KV_MXFP4, kv_scale=ops.PA_SCALE_E8M0_32, qlen=2,
                          kv_stride_token=64, kv_stride_head=64 * 128, kv_stride_block=64 * 128),
     ops.PA_ERR_UNSUPPORTED),
    ("unknown kv dtype", dict(kv_dtype=7), ops.PA_ERR_INVALID_ARG),
    ("merge flag not 0/1", dict(merge_in_decode=2), ops.PA_ERR_INVALID_ARG),
    ("negative sliding window", dict(sliding_window=-1), ops.PA_ERR_INVALID_ARG),
    ("trans_v not 0/1", dict(trans_v=2), ops.PA_ERR_INVALID_ARG),
    ("unknown kernel choice", dict(kernel=3), ops.PA_ERR_INVALID_ARG),
    ("negative kernel choice", dict(kernel=-1), ops.PA_ERR_INVALID_ARG),
    ("trans_v with per-token scales", dict(trans_v=1), ops.PA_ERR_UNSUPPORTED),
    ("trans_v with bf16", dict(trans_v=1, kv_dtype=ops.PA_KV_BF16, kv_scale=ops.PA_SCALE_NONE,
                               kv_stride_token=256, kv_stride_head=256 * 128,
                               kv_stride_block=256 * 128), ops.PA_ERR_UNSUPPORTED),
    ("null query", dict(query=None), ops.PA_ERR_INVALID_ARG),
    ("null scales", dict(key_scale=None), ops.PA_ERR_INVALID_ARG),
    ("e4m3 query without scale", dict(q_dtype=ops.PA_Q_FP8_E4M3), ops.PA_ERR_INVALID_ARG),
    ("non-dense token rows", dict(kv_stride_token=256, kv_stride_head=256 * 128,
                                  kv_stride_block=256 * 128), ops.PA_ERR_UNSUPPORTED),
    ("overlapping heads", dict(kv_stride_head=64), ops.PA_ERR_INVALID_ARG),
    ("unaligned head stride", dict(kv_stride_head=128 * 128 + 8, kv_stride_block=2 * 128 * 128),
     ops.PA_ERR_UNSUPPORTED),
    ("unaligned cache", dict(key_cache=(1 << 20) + 8), ops.PA_ERR_UNSUPPORTED),
    ("block table stride < width", dict(bt_stride=8), ops.PA_ERR_INVALID_ARG),
    ("short scale head stride", dict(scale_stride_head=16), ops.PA_ERR_INVALID_ARG),
    ("query head stride < D", dict(q_stride_head=64), ops.PA_ERR_INVALID_ARG),
    ("table span beyond 2^30 tokens", dict(max_blocks_per_seq=1 << 24, bt_stride=1 << 24),
     ops.PA_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("what,changes,status", REFUSED, ids=[r[0] for r in REFUSED])
def test_refused_arguments(lib, what, changes, status):
    a = _valid_args()
    for k, v in changes.items():
        setattr(a, k, v)
    assert ops.pa_decode_validate(a) == status
    assert lib.pa_decode_workspace_size(ctypes.byref(a)) == 0
    # every entry point refuses before touching the device
    for fn in ("pa_decode_plan", "pa_decode", "pa_decode_reduce", "pa_decode_run"):
        assert getattr(lib, fn)(ctypes.byref(a), 1 << 20, 1 << 30, None) == status


def test_workspace_too_small_is_refused(lib):
    a = _valid_args()
    n = ops.pa_decode_workspace_size(a)
    assert lib.pa_decode_plan(ctypes.byref(a), 1 << 20, n - 1, None) == ops.PA_ERR_WORKSPACE
    assert lib.pa_decode(ctypes.byref(a), (1 << 20) + 16, n, None) == ops.PA_ERR_WORKSPACE
    assert lib.pa_decode_reduce(ctypes.byref(a), None, n, None) == ops.PA_ERR_WORKSPACE


def test_workspace_grows_with_budget_and_rows(lib):
    a = _valid_args()
    n1 = ops.pa_decode_workspace_size(a)
    a.task_budget = 304
    n2 = ops.pa_decode_workspace_size(a)
    assert n2 > n1
    a.max_partitions = 1  # direct output needs no partial scratch
    n3 = ops.pa_decode_workspace_size(a)
    assert n3 < n1


def test_status_strings(lib):
    for s in (0, -1, -2, -3, -4):
        assert lib.pa_status_string(s)


def test_write_args_layout_matches_header():
    # 5 int32 (padded to 24 bytes), then 13 pointers and int64s
    assert ops.Mxfp4WriteArgs.key.offset == 24
    assert ops.Mxfp4WriteArgs.scale_stride_head.offset == 24 + 12 * 8
    assert ctypes.sizeof(ops.Mxfp4WriteArgs) == 24 + 13 * 8


def _valid_write_args():
    a = ops.Mxfp4WriteArgs()
    a.num_tokens, a.num_kv_heads, a.head_dim, a.page_size, a.num_blocks = 4, 2, 128, 128, 8
    fake = 1 << 20
    a.key, a.value, a.slot_mapping = fake, fake * 2, fake * 3
    a.src_stride_token, a.src_stride_head = 2 * 128, 128
    a.key_cache, a.value_cache = fake * 4, fake * 5
    a.cache_stride_head, a.cache_stride_block = 128 * 64, 2 * 128 * 64
    a.key_scale, a.value_scale = fake * 6, fake * 7
    a.scale_stride_head, a.scale_stride_block = 128 * 4, 2 * 128 * 4
    return a


WRITE_REFUSED = [
    ("head_dim 96", dict(head_dim=96), ops.PA_ERR_UNSUPPORTED),
    ("page 48", dict(page_size=48), ops.PA_ERR_UNSUPPORTED),
    ("no key", dict(key=None), ops.PA_ERR_INVALID_ARG),
    ("no slot mapping", dict(slot_mapping=None), ops.PA_ERR_INVALID_ARG),
    ("negative tokens", dict(num_tokens=-1), ops.PA_ERR_INVALID_ARG),
    ("overlapping source heads", dict(src_stride_head=64), ops.PA_ERR_INVALID_ARG),
    ("overlapping cache heads", dict(cache_stride_head=64), ops.PA_ERR_INVALID_ARG),
    ("short scale head stride", dict(scale_stride_head=8), ops.PA_ERR_INVALID_ARG),
    ("unaligned key", dict(key=(1 << 20) + 2), ops.PA_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("what,changes,status", WRITE_REFUSED, ids=[r[0] for r in WRITE_REFUSED])
def test_write_refused_arguments(lib, what, changes, status):
    a = _valid_write_args()
    for k, v in changes.items():
        setattr(a, k, v)
    assert lib.pa_mxfp4_kv_write(ctypes.byref(a), None) == status


def test_write_with_no_tokens_launches_nothing(lib):
    a = _valid_write_args()
    a.num_tokens = 0
    assert lib.pa_mxfp4_kv_write(ctypes.byref(a), None) == ops.PA_OK


def test_tensor_wrapper_refuses_host_tensors():
    # the one-call wrapper needs every tensor on one CUDA device (checked before any call)
    import torch
    q = torch.zeros(2, 1, 8, 128, dtype=torch.bfloat16)
    kc = torch.zeros(4, 1, 16, 128, dtype=torch.bfloat16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    ctx = torch.ones(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="one CUDA device"):
        ops.paged_attention_decode(q, kc, kc, bt, ctx)


def test_make_args_fills_the_variant_fields():
    # host tensors are enough: make_args reads shapes, strides and pointers only
    import torch
    B, qlen, Hq, Hkv, D, S, NB = 2, 3, 8, 2, 128, 16, 6
    q = torch.zeros(B, qlen, Hq, D, dtype=torch.bfloat16)
    kc = torch.zeros(NB, Hkv, S, D, dtype=torch.uint8)
    vt = torch.zeros(NB, Hkv, D, S, dtype=torch.uint8)  # transposed value cache
    bt = torch.zeros(B, 4, dtype=torch.int32)
    ctx = torch.ones(B, dtype=torch.int32)
    out = torch.empty(B, qlen, Hq, D, dtype=torch.bfloat16)
    sc = torch.tensor([0.05], dtype=torch.float32)
    sinks = torch.zeros(Hq, dtype=torch.float32)
    a = ops.make_args(q, kc, vt, bt, ctx, out, key_scale=sc, value_scale=sc, causal=True,
                      sliding_window=100, trans_v=True, sinks=sinks)
    assert (a.causal, a.sliding_window, a.trans_v) == (1, 100, 1)
    assert a.sinks == sinks.data_ptr() and a.kv_dtype == ops.PA_KV_FP8_E4M3
    assert a.kv_scale == ops.PA_SCALE_PER_TENSOR and a.qlen == qlen
    # a token-major value cache with trans_v, and sinks of the wrong size or type, are refused
    with pytest.raises(ValueError):
        ops.make_args(q, kc, kc, bt, ctx, out, key_scale=sc, value_scale=sc, trans_v=True)
    with pytest.raises(ValueError):
        ops.make_args(q, kc, kc, bt, ctx, out, key_scale=sc, value_scale=sc,
                      sinks=torch.zeros(Hq - 1))
    with pytest.raises(ValueError):
        ops.make_args(q, kc, kc, bt, ctx, out, key_scale=sc, value_scale=sc,
                      sinks=torch.zeros(Hq, dtype=torch.float64))


def _host_call(**over):
    """Host tensors of a small fp8 per-token call (make_args reads shapes and strides only)."""
    import torch
    B, qlen, Hq, Hkv, D, S, NB = 2, 1, 16, 1, 128, 16, 6
    t = dict(query=torch.zeros(B, qlen, Hq, D, dtype=torch.bfloat16),
             key_cache=torch.zeros(NB, Hkv, S, D, dtype=torch.uint8),
             value_cache=torch.zeros(NB, Hkv, S, D, dtype=torch.uint8),
             block_tables=torch.zeros(B, 4, dtype=torch.int32),
             context_lens=torch.ones(B, dtype=torch.int32),
             out=torch.empty(B, qlen, Hq, D, dtype=torch.bfloat16),
             key_scale=torch.ones(NB, Hkv, S, dtype=torch.float32),
             value_scale=torch.ones(NB, Hkv, S, dtype=torch.float32))
    t.update(over)
    return t


def _make(t, **kw):
    return ops.make_args(t["query"], t["key_cache"], t["value_cache"], t["block_tables"],
                         t["context_lens"], t["out"], key_scale=t["key_scale"],
                         value_scale=t["value_scale"], **kw)


def _bad_calls():
    import torch
    B, Hq, D, S, NB = 2, 16, 128, 16, 6
    return [
        ("out smaller than query", dict(out=torch.empty(B, 1, Hq, D // 2, dtype=torch.bfloat16))),
        ("out not bf16", dict(out=torch.empty(B, 1, Hq, D, dtype=torch.float32))),
        ("strided query head dim", dict(query=torch.zeros(B, 1, Hq, 2 * D, dtype=torch.bfloat16)[..., ::2])),
        ("strided out head dim", dict(out=torch.empty(B, 1, Hq, 2 * D, dtype=torch.bfloat16)[..., ::2])),
        ("int64 context lengths", dict(context_lens=torch.ones(B, dtype=torch.int64))),
        ("int64 block tables", dict(block_tables=torch.zeros(B, 4, dtype=torch.int64))),
        ("non-contiguous block tables", dict(block_tables=torch.zeros(4, B, dtype=torch.int32).t())),
        ("context lengths of another batch", dict(context_lens=torch.ones(B + 1, dtype=torch.int32))),
        ("block tables of another batch", dict(block_tables=torch.zeros(B + 1, 4, dtype=torch.int32))),
        ("key and value caches of different types",
         dict(value_cache=torch.zeros(NB, 1, S, D // 2, dtype=torch.bfloat16))),
        ("fp64 per-token scales", dict(key_scale=torch.ones(NB, 1, S, dtype=torch.float64),
                                        value_scale=torch.ones(NB, 1, S, dtype=torch.float64))),
        ("per-token scales of the wrong shape", dict(key_scale=torch.ones(NB, 1, S + 1),
                                                     value_scale=torch.ones(NB, 1, S + 1))),
        ("mxfp4 scales not uint8", dict(key_cache=torch.zeros(NB, 1, 128, D // 2, dtype=torch.uint8),
                                         value_cache=torch.zeros(NB, 1, 128, D // 2, dtype=torch.uint8),
                                         key_scale=torch.ones(NB, 1, 128, 4),
                                         value_scale=torch.ones(NB, 1, 128, 4))),
    ]


@pytest.mark.parametrize("what,over", _bad_calls(), ids=[c[0] for c in _bad_calls()])
def test_make_args_refuses_malformed_tensors(what, over):
    # each of these, passed on, would read or write out of bounds or read the wrong bytes
    with pytest.raises(ValueError):
        _make(_host_call(**over))


def test_make_args_kernel_choice():
    t = _host_call()
    assert _make(t).kernel == ops.PA_KERNEL_DEFAULT
    assert _make(t, kernel="mma").kernel == ops.PA_KERNEL_MMA
    assert _make(t, kernel="tc").kernel == ops.PA_KERNEL_TCGEN05
    with pytest.raises(ValueError):
        _make(t, kernel="triton")


def test_call_device_guard():
    # the one-call wrapper makes the tensors' device current; tensors spread over two devices,
    # or an explicit stream of another device, are refused before any launch (fakes carrying a
    # .device stand in for CUDA tensors and streams on this host)
    import types

    import torch
    d0, d1 = torch.device("cuda", 0), torch.device("cuda", 1)
    a, b = types.SimpleNamespace(device=d0), types.SimpleNamespace(device=d1)
    assert ops.call_device([a, None, a]) == d0
    assert ops.call_device([a], types.SimpleNamespace(device=d0)) == d0
    with pytest.raises(ValueError, match="one CUDA device"):
        ops.call_device([a, b])
    with pytest.raises(ValueError, match="stream is on"):
        ops.call_device([a, a], types.SimpleNamespace(device=d1))
