"""Helpers for the GPU parity tests: block buffers, inputs, oracle runs, comparisons.

Inputs come from the seeded generator (synth); expected values come from the
oracle on the host. Nothing here computes the update itself.
"""

from __future__ import annotations

import ctypes
from typing import Dict, List, Optional

import numpy as np

import oracle
import synth
from optimizer_update_gb300 import Layout, lst

SEED = synth.DEFAULT_SEED

# Hyperparameters of the workloads: AdamW lr 1e-4, betas 0.9 / 0.999, eps 1e-8,
# weight decay 0.01; the LoRA adapters use lr 2e-4 and no weight decay.
HP = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
HP_LORA = dict(lr=2e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)

F32_REL = 1e-6
F32_ABS = 1e-30


def hparams_for(workload: str, t: int):
    d = HP_LORA if workload.startswith("tinyllama_lora") else HP
    return lst.adamw_hparams(step=t, **d), oracle.hparams(step=t, **d)


def host_array(ptr: int, nbytes: int) -> np.ndarray:
    return np.ctypeslib.as_array((ctypes.c_uint8 * nbytes).from_address(ptr))


class PinnedBlocks:
    """One page-locked host block per layer (lst_host_alloc). With guard > 0
    (a multiple of 4096), each block sits between two canary bands of
    `guard` bytes inside its allocation; guards_intact() checks them."""

    def __init__(self, L: Layout, guard: int = 0):
        assert guard % 4096 == 0
        self.guard = guard
        self._allocs: List[int] = []
        self._full: List[np.ndarray] = []
        self.ptrs: List[int] = []
        self.arrays: List[np.ndarray] = []
        for i in range(L.n_layers):
            n = L.block_bytes(i)
            base = lst.lst_host_alloc(n + 2 * guard)
            self._allocs.append(base)
            if guard:
                full = host_array(base, n + 2 * guard)
                full[:guard] = 0xA5
                full[guard + n:] = 0x5A
                self._full.append(full)
            self.ptrs.append(base + guard)
            self.arrays.append(host_array(base + guard, n))

    def guards_intact(self) -> bool:
        g = self.guard
        return all(bool((f[:g] == 0xA5).all()) and bool((f[-g:] == 0x5A).all()) for f in self._full)

    def free(self) -> None:
        self.arrays = []
        self._full = []
        for p in self._allocs:
            lst.lst_host_free(p)
        self._allocs = []
        self.ptrs = []


def fill_host_block(L: Layout, i: int, arr: np.ndarray, workload: str, t: int, seed: int = SEED,
                    g_seed: Optional[int] = None) -> None:
    synth.fill_block(L.numpy_views(i, arr), L.spans(i), i, workload, L.fmt, t, seed, g_seed)


def redraw_gradient(L: Layout, i: int, arr: np.ndarray, workload: str, t: int, g_seed: int) -> None:
    """Write a fresh gradient (seed g_seed) into block i's G segment."""
    synth.fill_field(L.numpy_views(i, arr)["G"], "G", L.fmt, L.spans(i), i, workload, t, g_seed)


def device_blocks(L: Layout, guard: int = 0):
    """One device buffer per block; with guard > 0, the block sits between two
    canary bands of `guard` bytes. Returns (block tensors, backing tensors)."""
    import torch
    blocks, backing = [], []
    for i in range(L.n_layers):
        n = L.block_bytes(i)
        if guard:
            full = torch.empty(n + 2 * guard, dtype=torch.uint8, device="cuda")
            full[:guard].fill_(0xA5)
            full[guard + n:].fill_(0x5A)
            backing.append(full)
            blocks.append(full[guard:guard + n])
        else:
            b = torch.empty(n, dtype=torch.uint8, device="cuda")
            backing.append(b)
            blocks.append(b)
    return blocks, backing


def guards_intact(backing, L: Layout, guard: int) -> bool:
    for i, full in enumerate(backing):
        n = L.block_bytes(i)
        if not bool((full[:guard] == 0xA5).all()) or not bool((full[guard + n:] == 0x5A).all()):
            return False
    return True


def oracle_step(L: Layout, arr: np.ndarray, i: int, ohp, sgd: bool = False, threads: int = 8) -> None:
    oracle.step(L.fmt, L.numpy_views(i, arr), ohp, sgd=sgd, threads=threads)


OUTPUT_FIELDS = {"L12": ("W", "M", "V"), "L16M": ("MASTER", "M", "V", "W"), "L16F": ("W", "M", "V")}
FIELD_DT = {"L12": {"G": "bf16", "W": "bf16", "M": "f32", "V": "f32"},
            "L16M": {"G": "bf16", "MASTER": "f32", "M": "f32", "V": "f32", "W": "bf16"},
            "L16F": {"G": "f32", "W": "f32", "M": "f32", "V": "f32"}}


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between bit patterns (monotone integer order)."""
    def order(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(order(a) - order(b))


def compare(fmt: str, got: Dict[str, np.ndarray], exp: Dict[str, np.ndarray], fields=None) -> Dict[str, dict]:
    """Per-field check against the stated tolerances; returns stats and raises on failure.

    fp32 fields: |got - exp| <= 1e-6 |exp| + 1e-30 (NaN only where NaN).
    bf16 fields: within 1 bf16 ulp of the oracle's round-to-nearest-even result.
    """
    stats = {}
    for f in fields or OUTPUT_FIELDS[fmt]:
        g, e = got[f], exp[f]
        assert g.shape == e.shape, f
        if FIELD_DT[fmt][f] == "f32":
            gn, en = np.isnan(g), np.isnan(e)
            assert np.array_equal(gn, en), f"{f}: NaN pattern differs"
            ok = ~en
            err = np.abs(g[ok].astype(np.float64) - e[ok].astype(np.float64))
            lim = F32_REL * np.abs(e[ok].astype(np.float64)) + F32_ABS
            bad = np.nonzero(err > lim)[0]
            assert bad.size == 0, (f"{f}: {bad.size} elements outside 1e-6 rel; first at {bad[0]}: "
                                   f"got {g[ok][bad[0]]!r} expected {e[ok][bad[0]]!r}")
            exact = int(np.count_nonzero(g.view(np.uint32) == e.view(np.uint32)))
            stats[f] = dict(n=int(g.size), bit_exact=exact, max_rel=float((err / np.maximum(np.abs(
                e[ok].astype(np.float64)), 1e-300)).max()) if err.size else 0.0)
        else:
            d = bf16_ulp_distance(g, e)
            assert int(d.max(initial=0)) <= 1, f"{f}: bf16 differs by {int(d.max())} ulp"
            stats[f] = dict(n=int(g.size), bit_exact=int(np.count_nonzero(d == 0)), max_ulp=int(d.max(initial=0)))
    return stats


def sample_indices(padded: int, spans, rng: np.random.Generator, n_random: int = 8192) -> np.ndarray:
    """Block element indices to check at full size: both ends, tensor
    boundaries, padding, and a random sample."""
    idx = [np.arange(min(4096, padded)), np.arange(max(0, padded - 4096), padded)]
    for (_, off, n) in spans:
        for e in (off, off + n - 1, off + n):
            if 0 <= e < padded:
                idx.append(np.array([e]))
    idx.append(rng.integers(0, padded, size=n_random))
    return np.unique(np.concatenate(idx))


def gathered_inputs(L: Layout, i: int, workload: str, t: int, idx: np.ndarray, seed: int = SEED,
                    g_seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """The generator's input values of every field of block i at indices idx."""
    out = {}
    for f in FIELD_DT[L.fmt]:
        out[f] = np.ascontiguousarray(synth.gather_block(f, L.fmt, L.spans(i), i, workload, t, idx, seed, g_seed))
    return out


def gather_device(views, idx: np.ndarray) -> Dict[str, np.ndarray]:
    """Values of device field views (torch) at indices idx, as numpy arrays."""
    import torch
    ti = torch.from_numpy(idx.astype(np.int64)).to(views["G"].device)
    out = {}
    for f, v in views.items():
        x = v.index_select(0, ti).cpu().numpy()
        out[f] = x.view(np.uint16) if x.dtype == np.int16 else x
    return out
