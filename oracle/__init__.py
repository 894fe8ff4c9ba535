"""ORACLE - test infrastructure only.

Plain CPU statement of the packed-state AdamW / SGD update (``oracle.c``) and of
the packed block geometry (``layout.py``). Only the tests, the smoke check and
the bench's CPU-baseline leg import this package; the product library never
does, and the two share no code.

The numpy wrappers below only marshal arrays into the C loops. ``threads``
splits the element range into contiguous slices and runs the same C loop on
each slice from a Python thread (ctypes releases the GIL); the update is
elementwise, so the split does not change any result.
"""

from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


class Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64)]


class Scalars(ctypes.Structure):
    _fields_ = [("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("one_minus_beta1", ctypes.c_float), ("one_minus_beta2", ctypes.c_float),
                ("bias_correction1", ctypes.c_float), ("bias_correction2", ctypes.c_float),
                ("eps", ctypes.c_float), ("lr", ctypes.c_float), ("decay", ctypes.c_float)]


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            from . import build as _b
            _b.build()
        L = ctypes.CDLL(_LIB_PATH)
        i64, vp, f32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
        L.orc_make_scalars.argtypes = [ctypes.POINTER(Hparams), ctypes.POINTER(Scalars)]
        L.orc_make_scalars.restype = ctypes.c_int
        L.orc_adamw_l12.argtypes = [i64, vp, vp, vp, vp, ctypes.POINTER(Scalars)]
        L.orc_adamw_l16m.argtypes = [i64, vp, vp, vp, vp, vp, ctypes.POINTER(Scalars)]
        L.orc_adamw_l16f.argtypes = [i64, vp, vp, vp, vp, ctypes.POINTER(Scalars)]
        L.orc_sgd_l12.argtypes = [i64, vp, vp, f32]
        L.orc_sgd_l16m.argtypes = [i64, vp, vp, vp, f32]
        L.orc_sgd_l16f.argtypes = [i64, vp, vp, f32]
        L.orc_bf16_from_f32_array.argtypes = [i64, vp, vp]
        L.orc_f32_from_bf16_array.argtypes = [i64, vp, vp]
        L.orc_grad_sq_bf16.argtypes = [i64, vp]
        L.orc_grad_sq_bf16.restype = ctypes.c_double
        L.orc_grad_sq_f32.argtypes = [i64, vp]
        L.orc_grad_sq_f32.restype = ctypes.c_double
        for fn in ("orc_adamw_l12", "orc_adamw_l16m", "orc_adamw_l16f", "orc_sgd_l12", "orc_sgd_l16m",
                   "orc_sgd_l16f", "orc_bf16_from_f32_array", "orc_f32_from_bf16_array"):
            getattr(L, fn).restype = None
        _lib = L
    return _lib


def hparams(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1) -> Hparams:
    return Hparams(lr, beta1, beta2, eps, weight_decay, step)


def scalars(hp: Hparams) -> Scalars:
    s = Scalars()
    if lib().orc_make_scalars(ctypes.byref(hp), ctypes.byref(s)) != 0:
        raise ValueError("hyperparameters outside the method's domain")
    return s


def _check(a: np.ndarray, dtype, n: int, name: str) -> None:
    if a.dtype != dtype or not a.flags["C_CONTIGUOUS"] or a.size != n:
        raise TypeError(f"{name}: need contiguous {np.dtype(dtype).name}[{n}], got {a.dtype}[{a.size}]")


def _split(n: int, threads: Optional[int], fn, *arrays) -> None:
    """Run fn(count, *pointers) over [0, n) in contiguous slices."""
    t = max(1, int(threads or 1))
    if t == 1 or n < (1 << 16):
        fn(n, *[a.ctypes.data for a in arrays])
        return
    per = (n + t - 1) // t
    jobs = []
    for k in range(t):
        a, b = k * per, min(n, (k + 1) * per)
        if a >= b:
            break
        jobs.append((b - a, [x.ctypes.data + a * x.itemsize for x in arrays]))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        list(ex.map(lambda j: fn(j[0], *j[1]), jobs))


def adamw_l12(G, W, m, v, hp: Hparams, threads: Optional[int] = None) -> None:
    """In place: bf16 W (uint16), fp32 m, v; bf16 G read only."""
    n = G.size
    _check(G, np.uint16, n, "G"); _check(W, np.uint16, n, "W")
    _check(m, np.float32, n, "m"); _check(v, np.float32, n, "v")
    s = scalars(hp)
    _split(n, threads, lambda c, g, w, mm, vv: lib().orc_adamw_l12(c, g, w, mm, vv, ctypes.byref(s)),
           G, W, m, v)


def adamw_l16m(G, master, m, v, W, hp: Hparams, threads: Optional[int] = None) -> None:
    """In place: fp32 master, m, v; bf16 W written from the new master; bf16 G read only."""
    n = G.size
    _check(G, np.uint16, n, "G"); _check(master, np.float32, n, "master")
    _check(m, np.float32, n, "m"); _check(v, np.float32, n, "v"); _check(W, np.uint16, n, "W")
    s = scalars(hp)
    _split(n, threads,
           lambda c, g, ms, mm, vv, w: lib().orc_adamw_l16m(c, g, ms, mm, vv, w, ctypes.byref(s)),
           G, master, m, v, W)


def adamw_l16f(G, W, m, v, hp: Hparams, threads: Optional[int] = None) -> None:
    """In place: fp32 W, m, v; fp32 G read only."""
    n = G.size
    _check(G, np.float32, n, "G"); _check(W, np.float32, n, "W")
    _check(m, np.float32, n, "m"); _check(v, np.float32, n, "v")
    s = scalars(hp)
    _split(n, threads, lambda c, g, w, mm, vv: lib().orc_adamw_l16f(c, g, w, mm, vv, ctypes.byref(s)),
           G, W, m, v)


def sgd_l12(G, W, lr: float, threads: Optional[int] = None) -> None:
    n = G.size
    _check(G, np.uint16, n, "G"); _check(W, np.uint16, n, "W")
    _split(n, threads, lambda c, g, w: lib().orc_sgd_l12(c, g, w, lr), G, W)


def sgd_l16m(G, master, W, lr: float, threads: Optional[int] = None) -> None:
    n = G.size
    _check(G, np.uint16, n, "G"); _check(master, np.float32, n, "master"); _check(W, np.uint16, n, "W")
    _split(n, threads, lambda c, g, ms, w: lib().orc_sgd_l16m(c, g, ms, w, lr), G, master, W)


def sgd_l16f(G, W, lr: float, threads: Optional[int] = None) -> None:
    n = G.size
    _check(G, np.float32, n, "G"); _check(W, np.float32, n, "W")
    _split(n, threads, lambda c, g, w: lib().orc_sgd_l16f(c, g, w, lr), G, W)


def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.size, dtype=np.uint16)
    lib().orc_bf16_from_f32_array(x.size, x.ctypes.data, out.ctypes.data)
    return out.reshape(x.shape)


def f32_from_bf16(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.size, dtype=np.float32)
    lib().orc_f32_from_bf16_array(b.size, b.ctypes.data, out.ctypes.data)
    return out.reshape(b.shape)


def step(fmt: str, fields: dict, hp: Hparams, sgd: bool = False, threads: Optional[int] = None) -> None:
    """Apply one step to a block's field arrays (dict as produced by layout views)."""
    if fmt == "L12":
        if sgd:
            sgd_l12(fields["G"], fields["W"], hp.lr, threads)
        else:
            adamw_l12(fields["G"], fields["W"], fields["M"], fields["V"], hp, threads)
    elif fmt == "L16M":
        if sgd:
            sgd_l16m(fields["G"], fields["MASTER"], fields["W"], hp.lr, threads)
        else:
            adamw_l16m(fields["G"], fields["MASTER"], fields["M"], fields["V"], fields["W"], hp, threads)
    elif fmt == "L16F":
        if sgd:
            sgd_l16f(fields["G"], fields["W"], hp.lr, threads)
        else:
            adamw_l16f(fields["G"], fields["W"], fields["M"], fields["V"], hp, threads)
    else:
        raise ValueError(fmt)


def grad_sq(G: np.ndarray) -> float:
    """Sum of g^2 over a gradient array (bf16 bits as uint16, or fp32), in fp64."""
    G = np.ascontiguousarray(G)
    if G.dtype == np.uint16:
        return float(lib().orc_grad_sq_bf16(G.size, G.ctypes.data))
    if G.dtype == np.float32:
        return float(lib().orc_grad_sq_f32(G.size, G.ctypes.data))
    raise TypeError(G.dtype)
