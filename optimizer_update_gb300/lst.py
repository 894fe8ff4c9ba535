"""ctypes binding of liblst.so (include/lst.h), same names, argument marshalling only.

Every computation happens in the library's CUDA kernels and copy engines.
There is no fallback: if liblst.so has not been built, every call raises.
Pointers are plain Python ints (e.g. ``tensor.data_ptr()``); streams are
``cudaStream_t`` values as ints (e.g. ``torch.cuda.current_stream().cuda_stream``).
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblst.so")

# lst_status
LST_OK = 0
LST_ERR_INVALID_ARG = 1
LST_ERR_ALIGNMENT = 2
LST_ERR_NOT_PINNED = 3
LST_ERR_CUDA = 4
LST_ERR_OOM = 5
LST_ERR_TIMEOUT = 6
LST_ERR_IO = 7
# lst_format
LST_L12_BF16 = 0
LST_L16_MIXED = 1
LST_L16_FP32 = 2
# lst_field
LST_FIELD_G = 0
LST_FIELD_W = 1
LST_FIELD_M = 2
LST_FIELD_V = 3
LST_FIELD_MASTER = 4

FORMATS = {"L12": LST_L12_BF16, "L16M": LST_L16_MIXED, "L16F": LST_L16_FP32}
FIELDS = {"G": LST_FIELD_G, "W": LST_FIELD_W, "M": LST_FIELD_M, "V": LST_FIELD_V, "MASTER": LST_FIELD_MASTER}


class lst_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64)]


class lst_copy_choice(ctypes.Structure):
    _fields_ = [("measured", ctypes.c_int32), ("chunks", ctypes.c_int32), ("kernel_in_chunks", ctypes.c_int32),
                ("kernel_out_chunks", ctypes.c_int32), ("engine_h2d_gbs_min", ctypes.c_double),
                ("engine_h2d_gbs_max", ctypes.c_double), ("engine_d2h_gbs_min", ctypes.c_double),
                ("engine_d2h_gbs_max", ctypes.c_double)]


class lst_stream_stats(ctypes.Structure):
    _fields_ = [("steps_completed", ctypes.c_int64), ("h2d_bytes", ctypes.c_int64), ("d2h_bytes", ctypes.c_int64),
                ("chunks", ctypes.c_int32), ("kernel_in_chunks", ctypes.c_int32), ("kernel_out_chunks", ctypes.c_int32),
                ("timed", ctypes.c_int32), ("wall_ms", ctypes.c_double), ("h2d_busy_ms", ctypes.c_double),
                ("d2h_busy_ms", ctypes.c_double)]


class lst_step_options(ctypes.Structure):
    _fields_ = [("block_steps", ctypes.c_void_p), ("skip", ctypes.c_void_p), ("grad_sq", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p)]


def step_options(block_steps=None, skip=None, grad_sq: int = 0, workspace: int = 0):
    """Per-block options. block_steps / skip: sequences (host) of n_layers ints,
    or None; grad_sq / workspace: device pointers (ints) or 0. The returned
    structure keeps the host arrays alive."""
    o = lst_step_options()
    keep = []
    if block_steps is not None:
        a = (ctypes.c_int64 * max(1, len(block_steps)))(*[int(x) for x in block_steps])
        keep.append(a)
        o.block_steps = ctypes.cast(a, ctypes.c_void_p)
    if skip is not None:
        a = (ctypes.c_uint8 * max(1, len(skip)))(*[1 if x else 0 for x in skip])
        keep.append(a)
        o.skip = ctypes.cast(a, ctypes.c_void_p)
    o.grad_sq = grad_sq or None
    o.workspace = workspace or None
    o._keep = keep
    return o


def adamw_hparams(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1):
    return lst_adamw_hparams(lr, beta1, beta2, eps, weight_decay, step)


class LstError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [status {status}]")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load liblst.so; raises if it is not built (no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        i32, i64, vp, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
        P = ctypes.POINTER
        sig = {
            "lst_layout_create": ([i32, P(i32), P(i64), P(i32), ctypes.c_int, P(vp)], ctypes.c_int),
            "lst_layout_destroy": ([vp], None),
            "lst_layout_info": ([vp, P(i64), P(i64), P(i64)], ctypes.c_int),
            "lst_layout_block": ([vp, i64, P(i64), P(i64), P(i64)], ctypes.c_int),
            "lst_layout_segment": ([vp, i64, i32, P(i64), P(i64)], ctypes.c_int),
            "lst_layout_tensor": ([vp, i32, i32, P(i64), P(i64), P(i64)], ctypes.c_int),
            "lst_layout_transfer": ([vp, i64, P(i64), P(i64), P(i64), P(i64)], ctypes.c_int),
            "lst_layout_set_stream_chunk": ([vp, i64], ctypes.c_int),
            "lst_layout_set_stream_copy": ([vp, i32, i32], ctypes.c_int),
            "lst_stream_copy_choice": ([vp, i64, P(lst_copy_choice)], ctypes.c_int),
            "lst_stream_last_stats": ([vp, P(lst_stream_stats)], ctypes.c_int),
            "lst_adamw_step": ([vp, P(vp), P(lst_adamw_hparams), vp], ctypes.c_int),
            "lst_sgd_step": ([vp, P(vp), f32, vp], ctypes.c_int),
            "lst_stream_step": ([vp, P(vp), vp, vp, P(lst_adamw_hparams), i64], ctypes.c_int),
            "lst_zero_copy_step": ([vp, P(vp), P(lst_adamw_hparams), vp], ctypes.c_int),
            "lst_adamw_step_ex": ([vp, P(vp), P(lst_adamw_hparams), P(lst_step_options), vp], ctypes.c_int),
            "lst_stream_step_ex": ([vp, P(vp), vp, vp, P(lst_adamw_hparams), P(lst_step_options), i64],
                                   ctypes.c_int),
            "lst_workspace_bytes": ([], i64),
            "lst_stream_step_devgrad": ([vp, P(vp), P(vp), vp, vp, P(lst_adamw_hparams), P(lst_step_options), i64],
                                        ctypes.c_int),
            "lst_stream_step_devgrad_events": ([vp, P(vp), P(vp), P(vp), vp, vp, vp, P(lst_adamw_hparams),
                                                P(lst_step_options), i64], ctypes.c_int),
            "lst_adamw_step_ex_noalloc": ([vp, P(vp), P(lst_adamw_hparams), vp, vp, vp, vp], ctypes.c_int),
            "lst_host_alloc": ([i64, P(vp)], ctypes.c_int),
            "lst_host_free": ([vp], ctypes.c_int),
            "lst_store_create": ([vp, ctypes.c_char_p, P(vp), i64, P(vp)], ctypes.c_int),
            "lst_store_open": ([vp, ctypes.c_char_p, P(vp)], ctypes.c_int),
            "lst_store_close": ([vp], None),
            "lst_store_block_step": ([vp, i64, P(i64)], ctypes.c_int),
            "lst_store_read": ([vp, i64, vp], ctypes.c_int),
            "lst_store_write": ([vp, i64, vp, i64], ctypes.c_int),
            "lst_store_step": ([vp, P(vp), vp, vp, P(lst_adamw_hparams), i64], ctypes.c_int),
            "lst_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "lst_last_error": ([], ctypes.c_char_p),
            "lst_test_inject": ([i32, i64], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != LST_OK:
        msg = lib().lst_last_error().decode(errors="replace")
        raise LstError(status, f"{lib().lst_status_string(status).decode()}: {msg}")


def _ptr_array(ptrs: Sequence[int]):
    arr = (ctypes.c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = int(p) if p else None
    return arr


# ---------------------------------------------------------------------------
def lst_layout_create(shapes: Sequence[Sequence[int]], layer_of_tensor: Sequence[int], fmt) -> int:
    """shapes: one shape (0..4 dims) per tensor; returns the layout handle."""
    fmt = FORMATS.get(fmt, fmt)
    n = len(shapes)
    if len(layer_of_tensor) != n:
        raise ValueError("one block index per tensor")
    ndim = (ctypes.c_int32 * max(1, n))()
    dims = (ctypes.c_int64 * max(1, 4 * n))()
    lay = (ctypes.c_int32 * max(1, n))()
    for i, s in enumerate(shapes):
        ndim[i] = len(s)
        for k, d in enumerate(s[:4]):
            dims[4 * i + k] = int(d)
        if len(s) > 4:
            ndim[i] = len(s)  # rejected by the library
        lay[i] = int(layer_of_tensor[i])
    out = ctypes.c_void_p()
    _check(lib().lst_layout_create(n, ndim, dims, lay, int(fmt), ctypes.byref(out)))
    return out.value


def lst_layout_destroy(handle: int) -> None:
    lib().lst_layout_destroy(handle)


def lst_layout_info(handle: int) -> Tuple[int, int, int]:
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().lst_layout_info(handle, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def lst_layout_block(handle: int, layer: int) -> Tuple[int, int, int]:
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().lst_layout_block(handle, layer, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def lst_layout_segment(handle: int, layer: int, field) -> Tuple[int, int]:
    field = FIELDS.get(field, field)
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().lst_layout_segment(handle, layer, int(field), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def lst_layout_tensor(handle: int, tensor: int, field) -> Tuple[int, int, int]:
    field = FIELDS.get(field, field)
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().lst_layout_tensor(handle, tensor, int(field), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def lst_layout_transfer(handle: int, layer: int) -> Tuple[int, int, int, int]:
    v = [ctypes.c_int64() for _ in range(4)]
    _check(lib().lst_layout_transfer(handle, layer, *[ctypes.byref(x) for x in v]))
    return tuple(x.value for x in v)


def lst_layout_set_stream_chunk(handle: int, elems: int) -> None:
    _check(lib().lst_layout_set_stream_chunk(handle, elems))


LST_COPY_ENGINE, LST_COPY_SM, LST_COPY_AUTO = 0, 1, 2


def lst_layout_set_stream_copy(handle: int, h2d_mode: int, d2h_mode: int) -> None:
    _check(lib().lst_layout_set_stream_copy(handle, h2d_mode, d2h_mode))


def lst_stream_copy_choice(handle: int, block: int) -> dict:
    """What LST_COPY_AUTO has learned about `block`: whether a streamed step
    timed it, its sub-chunks, how many of them later steps move with the copy
    kernel each way, and the copy-engine rates timed (GB/s, 0 where none)."""
    c = lst_copy_choice()
    _check(lib().lst_stream_copy_choice(handle, block, ctypes.byref(c)))
    return {f: (bool(getattr(c, f)) if f == "measured" else getattr(c, f)) for f, _ in c._fields_}


def lst_stream_last_stats(handle: int) -> dict:
    """The last completed streamed step on this layout: bytes moved each way,
    sub-chunks (and how many the copy kernel moved), host wall time and, when
    timed, the summed copy durations each way (ms)."""
    st = lst_stream_stats()
    _check(lib().lst_stream_last_stats(handle, ctypes.byref(st)))
    return {f: getattr(st, f) for f, _ in st._fields_}


def lst_adamw_step(handle: int, dev_blocks: Sequence[int], hparams: lst_adamw_hparams, stream: int = 0) -> None:
    _check(lib().lst_adamw_step(handle, _ptr_array(dev_blocks), ctypes.byref(hparams), stream or None))


def lst_sgd_step(handle: int, dev_blocks: Sequence[int], lr: float, stream: int = 0) -> None:
    _check(lib().lst_sgd_step(handle, _ptr_array(dev_blocks), lr, stream or None))


def lst_stream_step(handle: int, host_blocks: Sequence[int], dev_buf0: int, dev_buf1: int,
                    hparams: lst_adamw_hparams, timeout_ms: int = 0) -> None:
    _check(lib().lst_stream_step(handle, _ptr_array(host_blocks), dev_buf0, dev_buf1, ctypes.byref(hparams),
                                 timeout_ms))


def lst_zero_copy_step(handle: int, host_blocks: Sequence[int], hparams: lst_adamw_hparams,
                       stream: int = 0) -> None:
    _check(lib().lst_zero_copy_step(handle, _ptr_array(host_blocks), ctypes.byref(hparams), stream or None))


def lst_workspace_bytes() -> int:
    return int(lib().lst_workspace_bytes())


def lst_adamw_step_ex(handle: int, dev_blocks: Sequence[int], hparams: lst_adamw_hparams, opts=None,
                      stream: int = 0) -> None:
    _check(lib().lst_adamw_step_ex(handle, _ptr_array(dev_blocks), ctypes.byref(hparams),
                                   ctypes.byref(opts) if opts is not None else None, stream or None))


def lst_adamw_step_ex_noalloc(handle: int, dev_blocks: Sequence[int], hparams: lst_adamw_hparams,
                              block_steps=None, skip=None, grad_sq: int = 0, stream: int = 0) -> None:
    """The extended step using the library's own static scratch (no allocation)."""
    bs = (ctypes.c_int64 * max(1, len(block_steps)))(*[int(x) for x in block_steps]) if block_steps is not None else None
    sk = (ctypes.c_uint8 * max(1, len(skip)))(*[1 if x else 0 for x in skip]) if skip is not None else None
    _check(lib().lst_adamw_step_ex_noalloc(handle, _ptr_array(dev_blocks), ctypes.byref(hparams),
                                           ctypes.cast(bs, ctypes.c_void_p) if bs is not None else None,
                                           ctypes.cast(sk, ctypes.c_void_p) if sk is not None else None,
                                           grad_sq or None, stream or None))


def lst_stream_step_ex(handle: int, host_blocks: Sequence[int], dev_buf0: int, dev_buf1: int,
                       hparams: lst_adamw_hparams, opts=None, timeout_ms: int = 0) -> None:
    _check(lib().lst_stream_step_ex(handle, _ptr_array(host_blocks), dev_buf0, dev_buf1, ctypes.byref(hparams),
                                    ctypes.byref(opts) if opts is not None else None, timeout_ms))


def lst_stream_step_devgrad(handle: int, host_blocks: Sequence[int], dev_grads: Sequence[int], dev_buf0: int,
                            dev_buf1: int, hparams: lst_adamw_hparams, opts=None, timeout_ms: int = 0) -> None:
    _check(lib().lst_stream_step_devgrad(handle, _ptr_array(host_blocks), _ptr_array(dev_grads), dev_buf0, dev_buf1,
                                         ctypes.byref(hparams), ctypes.byref(opts) if opts is not None else None,
                                         timeout_ms))


def lst_stream_step_devgrad_events(handle: int, host_blocks: Sequence[int], dev_grads: Sequence[int],
                                   grad_ready: Sequence[int], order, dev_buf0: int, dev_buf1: int,
                                   hparams: lst_adamw_hparams, opts=None, timeout_ms: int = 0) -> None:
    """grad_ready: cudaEvent_t values as ints (0 for a gradient already
    complete), e.g. torch.cuda.Event.cuda_event; order: block indices or None."""
    ords = (ctypes.c_int64 * max(1, len(order)))(*[int(x) for x in order]) if order is not None else None
    _check(lib().lst_stream_step_devgrad_events(handle, _ptr_array(host_blocks), _ptr_array(dev_grads),
                                                _ptr_array(grad_ready),
                                                ctypes.cast(ords, ctypes.c_void_p) if ords is not None else None,
                                                dev_buf0, dev_buf1, ctypes.byref(hparams),
                                                ctypes.byref(opts) if opts is not None else None, timeout_ms))


def lst_store_create(layout: int, directory: str, host_blocks=None, step: int = 0) -> int:
    out = ctypes.c_void_p()
    hb = _ptr_array(host_blocks) if host_blocks is not None else None
    _check(lib().lst_store_create(layout, directory.encode(), hb, step, ctypes.byref(out)))
    return out.value


def lst_store_open(layout: int, directory: str) -> int:
    out = ctypes.c_void_p()
    _check(lib().lst_store_open(layout, directory.encode(), ctypes.byref(out)))
    return out.value


def lst_store_close(store: int) -> None:
    lib().lst_store_close(store)


def lst_store_block_step(store: int, layer: int) -> int:
    v = ctypes.c_int64()
    _check(lib().lst_store_block_step(store, layer, ctypes.byref(v)))
    return v.value


def lst_store_read(store: int, layer: int, host_dst: int) -> None:
    _check(lib().lst_store_read(store, layer, host_dst))


def lst_store_write(store: int, layer: int, host_src: int, step: int) -> None:
    _check(lib().lst_store_write(store, layer, host_src, step))


def lst_store_step(store: int, staging: Sequence[int], dev_buf0: int, dev_buf1: int, hparams: lst_adamw_hparams,
                   timeout_ms: int = 0) -> None:
    _check(lib().lst_store_step(store, _ptr_array(staging), dev_buf0, dev_buf1, ctypes.byref(hparams), timeout_ms))


def lst_host_alloc(nbytes: int) -> int:
    out = ctypes.c_void_p()
    _check(lib().lst_host_alloc(nbytes, ctypes.byref(out)))
    return out.value


def lst_host_free(ptr: int) -> None:
    _check(lib().lst_host_free(ptr))


def lst_status_string(status: int) -> str:
    return lib().lst_status_string(status).decode()


def lst_last_error() -> str:
    return lib().lst_last_error().decode(errors="replace")


def lst_test_inject(kind: int, k: int = 0) -> None:
    _check(lib().lst_test_inject(kind, k))
