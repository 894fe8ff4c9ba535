"""Seeded synthetic inputs for the packed-state optimizer: shapes and values.

This module is shared by the tests, the bench and the oracle's callers. It
holds no optimizer arithmetic: it draws input fields (weights, gradients, Adam
moments, master weights) for given tensor spans of a block and writes them
into caller-provided numpy arrays. Layout geometry (where each tensor sits) is
passed in by the caller.

The value definition (counter-based splitmix64 hash, variance-matched
Irwin-Hall(4) lattice stand-in for N(0, sigma), bf16 by truncation) is stated
in ``gen.c``.
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Dict, Iterable, List, Sequence, Tuple

import numpy as np

from . import shapes  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_DEV_LIB_PATH = os.path.join(_HERE, "libsynth_dev.so")
_lib = None
_dev_lib = None

# Field codes used in stream ids.
FIELD_W, FIELD_G, FIELD_M, FIELD_V, FIELD_MASTER = 1, 2, 3, 4, 5
FIELD_CODES = {"W": FIELD_W, "G": FIELD_G, "M": FIELD_M, "V": FIELD_V, "MASTER": FIELD_MASTER}

KIND_F32, KIND_BF16, KIND_SQ_F32 = 0, 1, 2

DEFAULT_SEED = 0x5EED

# Irwin-Hall(4) over 16-bit uniforms: variance of the centred sum.
_IH_SD = math.sqrt((2.0 ** 32 - 1.0) / 3.0)


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            from . import build as _b
            _b.build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, i64, f32, vp, ci = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
        for name in ("synth_fill_f32", "synth_fill_bf16", "synth_fill_sq_f32"):
            fn = getattr(L, name)
            fn.argtypes = [u64, u64, u64, i64, f32, vp, ci]
            fn.restype = ci
        L.synth_hash.argtypes = [u64, u64, u64]
        L.synth_hash.restype = u64
        L.synth_gather.argtypes = [ci, u64, u64, vp, i64, f32, vp]
        L.synth_gather.restype = ci
        _lib = L
    return _lib


def dev_lib():
    """The generator on the GPU (gen_dev.cu): a gradient producer that stands
    in for a backward pass. Raises if it has not been built."""
    global _dev_lib
    if _dev_lib is None:
        if not os.path.exists(_DEV_LIB_PATH):
            raise RuntimeError(f"{_DEV_LIB_PATH} is missing: run synth.build.build()")
        L = ctypes.CDLL(_DEV_LIB_PATH)
        u64, i64, f32, vp, ci = ctypes.c_uint64, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
        L.synth_dev_fill.argtypes = [ci, u64, u64, u64, i64, f32, vp, ci, vp]
        L.synth_dev_fill.restype = ci
        L.synth_dev_zero.argtypes = [vp, i64, vp]
        L.synth_dev_zero.restype = ci
        _dev_lib = L
    return _dev_lib


def scale_for(sigma: float) -> np.float32:
    """fp32 multiplier that maps the centred lattice draw to standard deviation sigma."""
    return np.float32(sigma / _IH_SD)


def stream_id(field: int, layer: int) -> int:
    return (int(field) << 32) | int(layer)


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def fill(out: np.ndarray, kind: int, seed: int, stream: int, start: int, sigma: float,
         threads: int | None = None) -> None:
    """Write values start .. start+out.size-1 of the stream into ``out`` (contiguous)."""
    if not out.flags["C_CONTIGUOUS"]:
        raise ValueError("fill needs a contiguous output array")
    want = np.uint16 if kind == KIND_BF16 else np.float32
    if out.dtype != want:
        raise TypeError(f"kind {kind} writes {want}, got {out.dtype}")
    fn = {KIND_F32: lib().synth_fill_f32, KIND_BF16: lib().synth_fill_bf16,
          KIND_SQ_F32: lib().synth_fill_sq_f32}[kind]
    rc = fn(seed & (2 ** 64 - 1), stream, start, out.size, float(scale_for(sigma)),
            out.ctypes.data, threads or _threads())
    if rc != 0:
        raise RuntimeError("synth fill failed")


def gather(kind: int, seed: int, stream: int, idx: np.ndarray, sigma: float) -> np.ndarray:
    """Values of the stream at the given indices (random access)."""
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.size, dtype=np.uint16 if kind == KIND_BF16 else np.float32)
    rc = lib().synth_gather(kind, seed & (2 ** 64 - 1), stream, idx.ctypes.data, idx.size,
                            float(scale_for(sigma)), out.ctypes.data)
    if rc != 0:
        raise RuntimeError("synth gather failed")
    return out


# ---------------------------------------------------------------------------
# Recipes: which distribution each field of each workload is drawn from.
# ---------------------------------------------------------------------------
# N(0, 0.02) weights, N(0, 1e-3) gradients, N(0, 1e-4) first moment and
# (N(0, 1e-3))^2 second moment; first and second moments are zero at t = 1.
STANDARD = {
    "W": ("normal", 0.02),
    "MASTER": ("normal", 0.02),
    "G": ("normal", 1e-3),
    "M": ("normal", 1e-4),
    "V": ("sq", 1e-3),
}

# Fields of each format, in block order, with their element dtype.
FORMAT_FIELDS = {
    "L12": (("G", "bf16"), ("W", "bf16"), ("M", "f32"), ("V", "f32")),
    "L16M": (("G", "bf16"), ("MASTER", "f32"), ("M", "f32"), ("V", "f32"), ("W", "bf16")),
    "L16F": (("G", "f32"), ("W", "f32"), ("M", "f32"), ("V", "f32")),
}


def field_dist(workload: str, field: str, tensor_name: str, t: int) -> Tuple[str, float]:
    """(kind, sigma) of a field for a tensor at step t. kind: normal | sq | zero."""
    if field in ("M", "V") and t <= 1:
        return ("zero", 0.0)
    if workload.startswith("tinyllama_lora") and field == "W" and tensor_name.endswith("lora_B"):
        return ("zero", 0.0) if t <= 1 else ("normal", 1e-3)
    return STANDARD[field]


def _kind(dist: str, dtype: str) -> int:
    if dist == "sq":
        return KIND_SQ_F32
    return KIND_BF16 if dtype == "bf16" else KIND_F32


def fill_field(arr: np.ndarray, field: str, fmt: str, spans: Sequence[Tuple[str, int, int]], layer: int,
               workload: str, t: int, seed: int = DEFAULT_SEED, threads: int | None = None) -> None:
    """Fill one field array of a block (padding set to zero)."""
    dtype = dict(FORMAT_FIELDS[fmt])[field]
    arr[...] = 0
    if fmt == "L16M" and field == "W":
        return  # the mixed layout's bf16 W is an output derived from MASTER
    for (name, off, n) in spans:
        if n == 0:
            continue
        dist, sigma = field_dist(workload, field, name, t)
        if dist == "zero":
            continue
        fill(arr[off:off + n], _kind(dist, dtype), seed, stream_id(FIELD_CODES[field], layer), off, sigma,
             threads)


def fill_block(fields: Dict[str, np.ndarray], spans: Sequence[Tuple[str, int, int]], layer: int,
               workload: str, fmt: str, t: int, seed: int = DEFAULT_SEED,
               g_seed: int | None = None, threads: int | None = None) -> None:
    """Fill every field array of one block.

    fields: field name -> 1-D array over the block's padded element space
            (uint16 for bf16 fields, float32 otherwise).
    spans:  (tensor_name, element_offset, numel) of every tensor in the block.
    Padding elements are set to zero. g_seed, if given, replaces the seed of the
    gradient field (a fresh gradient per step).
    """
    for field, _ in FORMAT_FIELDS[fmt]:
        s = g_seed if (field == "G" and g_seed is not None) else seed
        fill_field(fields[field], field, fmt, spans, layer, workload, t, s, threads)


def gather_block(field: str, fmt: str, spans: Sequence[Tuple[str, int, int]], layer: int,
                 workload: str, t: int, idx: np.ndarray, seed: int = DEFAULT_SEED,
                 g_seed: int | None = None) -> np.ndarray:
    """Input values of one field at block element indices idx (padding gives 0).

    The result equals ``fill_block``'s array for that field at those indices.
    """
    dtype = dict(FORMAT_FIELDS[fmt])[field]
    idx = np.asarray(idx, dtype=np.int64)
    out = np.zeros(idx.size, dtype=np.uint16 if dtype == "bf16" else np.float32)
    if fmt == "L16M" and field == "W":
        return out
    for (name, off, n) in spans:
        sel = np.nonzero((idx >= off) & (idx < off + n))[0]
        if sel.size == 0:
            continue
        dist, sigma = field_dist(workload, field, name, t)
        if dist == "zero":
            continue
        s = g_seed if (field == "G" and g_seed is not None) else seed
        out[sel] = gather(_kind(dist, dtype), s, stream_id(FIELD_CODES[field], layer), idx[sel], sigma)
    return out


def device_fill_field(dev_ptr: int, field: str, fmt: str, spans: Sequence[Tuple[str, int, int]], padded: int,
                      layer: int, workload: str, t: int, seed: int = DEFAULT_SEED, stream: int = 0,
                      passes: int = 1) -> None:
    """The GPU twin of fill_field: one field of a block written into device
    memory at dev_ptr (padded elements; padding and zero-valued tensors set to
    zero), enqueued on the CUDA stream `stream` (a cudaStream_t as an int).
    passes > 1 adds hash rounds per element that stand in for the compute of
    a backward pass; the values do not depend on it."""
    dtype = dict(FORMAT_FIELDS[fmt])[field]
    esz = 2 if dtype == "bf16" else 4
    L = dev_lib()
    rc = L.synth_dev_zero(dev_ptr, padded * esz, stream or None)
    if rc != 0:
        raise RuntimeError(f"synth_dev_zero failed ({rc})")
    if fmt == "L16M" and field == "W":
        return
    for (name, off, n) in spans:
        if n == 0:
            continue
        dist, sigma = field_dist(workload, field, name, t)
        if dist == "zero":
            continue
        rc = L.synth_dev_fill(_kind(dist, dtype), seed & (2 ** 64 - 1), stream_id(FIELD_CODES[field], layer), off,
                              n, float(scale_for(sigma)), dev_ptr + off * esz, int(passes), stream or None)
        if rc != 0:
            raise RuntimeError(f"synth_dev_fill failed ({rc})")
