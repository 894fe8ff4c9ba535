"""Streamed step (pinned host blocks, two device buffers, three streams) (GB300).

The streamed path runs the same kernel on the same bytes, so it must be
bit-identical to the device-resident path; it is also checked against the
oracle. Failure handling is exercised on the host only: a pageable block, a
host-side injected enqueue failure, and a completion that is never observed
(host deadline). No device fault is ever provoked.
"""

import time

import numpy as np
import pytest

import oracle
from optimizer_update_gb300 import Layout, lst
from synth import shapes

from gpu_util import (PinnedBlocks, compare, fill_host_block, gathered_inputs, hparams_for, oracle_step,
                      redraw_gradient, sample_indices)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    lst.lst_test_inject(0, 0)
    yield
    lst.lst_test_inject(0, 0)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _bufs(L):
    b0 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
    b1 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
    return b0, b1


def _stream_vs_device(specs, fmt, workload, t, chunk, steps=1, copy=None):
    L = Layout(specs, fmt)
    L.set_stream_chunk(chunk)
    if copy is not None:
        L.set_stream_copy(*copy)
    P = PinnedBlocks(L)
    try:
        for i in range(L.n_layers):
            fill_host_block(L, i, P.arrays[i], workload, t)
        dev = [torch.from_numpy(P.arrays[i].copy()).cuda() for i in range(L.n_layers)]
        ref = [P.arrays[i].copy() for i in range(L.n_layers)]
        b0, b1 = _bufs(L)
        for s in range(steps):
            hp, ohp = hparams_for(workload, t + s)
            lst.lst_adamw_step(L.handle, [d.data_ptr() for d in dev], hp, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), hp, 600_000)
            for i in range(L.n_layers):
                oracle_step(L, ref[i], i, ohp)
        for i in range(L.n_layers):
            d = dev[i].cpu().numpy()
            # streamed == device-resident, every byte (G included: read-only)
            assert np.array_equal(P.arrays[i], d), f"block {i}: streamed differs from device-resident"
            compare(fmt, L.numpy_views(i, P.arrays[i]), L.numpy_views(i, ref[i]))
    finally:
        P.free()
    return L


FMTS = [("L12", "tinyllama_layer_l12"), ("L16M", "tinyllama_full_l16m"), ("L16F", "tinyllama_lora_l16f")]


def _three_tinyllama_layers():
    specs = [(n, sh, l - 1) for (n, sh, l) in shapes.tinyllama_full() if l in (1, 2, 3)]
    return specs + [("odd", (4097,), 1), ("odder", (9,), 2)]


@pytest.mark.parametrize("fmt,workload", FMTS)
@pytest.mark.parametrize("chunk", [0, 1 << 20])
def test_stream_bit_identical_tinyllama_layers(fmt, workload, chunk):
    _stream_vs_device(_three_tinyllama_layers(), fmt, workload, 10, chunk, steps=2)


@pytest.mark.parametrize("fmt,workload", FMTS)
@pytest.mark.parametrize("chunk", [2048, 6144])
def test_stream_bit_identical_small_chunks(fmt, workload, chunk):
    specs = [("a", (70_001,), 0), ("b", (4097,), 1), ("c", (30_000,), 1), ("d", (9,), 2), ("e", (2048,), 3),
             ("f", (12_288,), 4)]
    _stream_vs_device(specs, fmt, workload, 3, chunk, steps=3)


E, SM, AUTO = lst.LST_COPY_ENGINE, lst.LST_COPY_SM, lst.LST_COPY_AUTO


@pytest.mark.parametrize("fmt,workload", FMTS)
@pytest.mark.parametrize("copy", [(E, E), (SM, E), (E, SM), (SM, SM)], ids=["ce-ce", "sm-ce", "ce-sm", "sm-sm"])
def test_stream_copy_modes_bit_identical(fmt, workload, copy):
    """Sub-chunks moved by the copy engines or by the SM copy kernel, in either
    direction: the same bytes as the device-resident step."""
    _stream_vs_device(_three_tinyllama_layers(), fmt, workload, 10, 1 << 20, steps=2, copy=copy)


@pytest.mark.parametrize("fmt,workload", FMTS)
@pytest.mark.parametrize("chunk", [0, 6144])
def test_stream_sm_copies_whole_blocks_and_ragged_chunks(fmt, workload, chunk):
    specs = [("a", (70_001,), 0), ("b", (4097,), 1), ("c", (30_000,), 1), ("d", (9,), 2), ("e", (2048,), 3)]
    _stream_vs_device(specs, fmt, workload, 3, chunk, steps=2, copy=(SM, SM))


# ---- LST_COPY_AUTO (the default): every copy-engine sub-chunk copy of a step
# is timed; a sub-chunk moved at under 0.4 of the best rate goes through the
# copy kernel in the later steps


def _auto_state(L):
    return [L.stream_copy_choice(i) for i in range(L.n_layers)]


@pytest.mark.parametrize("fmt,workload", FMTS)
def test_stream_auto_copy_default_bit_identical(fmt, workload):
    """The default mode, two steps: the same bytes as the device-resident
    step; every block timed, with positive rates each way (its sub-chunks
    are 12 MB or more)."""
    L = _stream_vs_device(_three_tinyllama_layers(), fmt, workload, 10, 1 << 20, steps=2)
    st = L.stream_last_stats()
    assert st["steps_completed"] == 2 and st["timed"] == 1, st
    assert st["h2d_bytes"] == sum(L.transfer(i)[1] for i in range(L.n_layers)), st
    assert st["d2h_bytes"] == sum(L.transfer(i)[3] for i in range(L.n_layers)), st
    assert st["chunks"] == sum(c["chunks"] for c in _auto_state(L)), st
    # each direction's copies run one after another on their stream
    for d in ("h2d", "d2h"):
        assert 0 < st[f"{d}_busy_ms"] <= 1.05 * st["wall_ms"] + 0.5, st
    for i, c in enumerate(_auto_state(L)):
        assert c["measured"] and c["chunks"] >= 1, (i, c)
        assert c["kernel_in_chunks"] <= c["chunks"] and c["kernel_out_chunks"] <= c["chunks"]
        if c["kernel_in_chunks"] < c["chunks"]:
            assert 0 < c["engine_h2d_gbs_min"] <= c["engine_h2d_gbs_max"], (i, c)
        if c["kernel_out_chunks"] < c["chunks"]:
            assert 0 < c["engine_d2h_gbs_min"] <= c["engine_d2h_gbs_max"], (i, c)


@pytest.mark.parametrize("fmt,workload", FMTS)
def test_stream_auto_copy_moves_slow_chunks_with_the_kernel(fmt, workload):
    """Blocks 0 and 2 seen as 100x slower on the copy engines in the first
    step (host-side test hook: nothing is slowed): the second step moves
    their sub-chunks of 4 MB or more with the copy kernel, both ways, and the
    bytes are those of the device-resident step; setting the mode again
    forgets what was learned. (Block 1 is not checked: on the shared hosts
    here a pinned allocation can really be slow on the copy engines in
    places, after other tests have pinned and freed a lot of memory, and then
    its slow sub-chunks rightly move with the copy kernel too.)"""
    lst.lst_test_inject(4, 2)
    L = _stream_vs_device(_three_tinyllama_layers(), fmt, workload, 10, 1 << 20, steps=2)
    st = _auto_state(L)
    for i in (0, 2):  # all but the step's short first (block 0) or last (block 2) sub-chunks under 4 MB
        assert st[i]["measured"] and st[i]["chunks"] > 4, (i, st[i])
        assert st[i]["chunks"] - 3 <= st[i]["kernel_in_chunks"] <= st[i]["chunks"], (i, st[i])
        assert st[i]["chunks"] - 3 <= st[i]["kernel_out_chunks"] <= st[i]["chunks"], (i, st[i])
    assert st[1]["measured"] and st[1]["chunks"] > 4, st[1]
    lst.lst_test_inject(0, 0)
    L.set_stream_copy(AUTO, AUTO)
    assert not L.stream_copy_choice(0)["measured"]


def test_stream_lora_many_small_blocks():
    _stream_vs_device(shapes.tinyllama_lora(), "L16F", "tinyllama_lora_l16f", 1, 1 << 16, steps=2)


@pytest.mark.slow
def test_stream_tinyllama_full_l16m_bit_identical():
    # TinyLlama-1.1B, 16 B/param mixed, 24 blocks, 17.6 GB pinned: one step
    _stream_vs_device(shapes.tinyllama_full(), "L16M", "tinyllama_full_l16m", 1, 1 << 22, steps=1)


@pytest.mark.slow
def test_stream_llama70b_slice_three_steps_sampled():
    """Llama-70B depth slice (8 x 855.6M params, 12 B/param, 82 GB pinned):
    t = 1..3 streamed, a fresh gradient per step drawn with seed + t; sampled
    elements followed through the three steps by the oracle."""
    workload, fmt = "llama70b_slice8_l12", "L12"
    L = Layout(shapes.llama70b_slice(8), fmt)
    P = PinnedBlocks(L)
    try:
        rng = np.random.default_rng(4)
        idx = [sample_indices(L.padded(i), L.spans(i), rng, 4096) for i in range(L.n_layers)]
        seed = 0x5EED
        for i in range(L.n_layers):
            fill_host_block(L, i, P.arrays[i], workload, 1, seed, g_seed=seed + 1)
        state = [gathered_inputs(L, i, workload, 1, idx[i], seed, g_seed=seed + 1) for i in range(L.n_layers)]
        b0, b1 = _bufs(L)
        for t in (1, 2, 3):
            if t > 1:  # a fresh gradient per step, drawn with seed + t
                for i in range(L.n_layers):
                    redraw_gradient(L, i, P.arrays[i], workload, t, seed + t)
                    state[i]["G"] = gathered_inputs(L, i, workload, t, idx[i], seed, g_seed=seed + t)["G"]
            hp, ohp = hparams_for(workload, t)
            t0 = time.time()
            lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), hp, 600_000)
            assert time.time() - t0 < 600
            for i in range(L.n_layers):
                oracle.step(fmt, state[i], ohp)
        for i in range(L.n_layers):
            got = {f: L.numpy_views(i, P.arrays[i])[f][idx[i]] for f in ("W", "M", "V")}
            s = compare(fmt, got, state[i])
            for f, d in s.items():
                assert d["bit_exact"] == d["n"], f
    finally:
        P.free()


# ---- failure handling (host side only) -------------------------------------
def _small():
    L = Layout([("a", (70_000,), 0), ("b", (50_000,), 1), ("c", (9,), 2)], "L12")
    L.set_stream_chunk(16384)
    return L


def test_not_pinned_is_rejected():
    L = _small()
    import ctypes
    pageable = [np.zeros(L.block_bytes(i) + 8192, np.uint8) for i in range(L.n_layers)]
    ptrs = [(a.ctypes.data + 4095) // 4096 * 4096 for a in pageable]
    b0, b1 = _bufs(L)
    with pytest.raises(lst.LstError) as e:
        lst.lst_stream_step(L.handle, ptrs, b0.data_ptr(), b1.data_ptr(), lst.adamw_hparams(), 10_000)
    assert e.value.status == lst.LST_ERR_NOT_PINNED


def test_host_pointer_as_device_buffer_is_rejected():
    L = _small()
    P = PinnedBlocks(L)
    try:
        b0, _ = _bufs(L)
        with pytest.raises(lst.LstError) as e:
            lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), P.ptrs[0], lst.adamw_hparams(), 10_000)
        assert e.value.status == lst.LST_ERR_INVALID_ARG
    finally:
        P.free()


@pytest.mark.parametrize("k", [1, 5, 23])
def test_injected_enqueue_failure_drains_and_recovers(k):
    L = _small()
    P = PinnedBlocks(L)
    try:
        for i in range(L.n_layers):
            fill_host_block(L, i, P.arrays[i], "fault", 2)
        b0, b1 = _bufs(L)
        lst.lst_test_inject(1, k)
        with pytest.raises(lst.LstError) as e:
            lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), lst.adamw_hparams(step=2), 60_000)
        assert e.value.status == lst.LST_ERR_CUDA and "injected" in str(e.value)
        lst.lst_test_inject(0, 0)
        # the context and the engine are still usable: a clean step from a fresh state matches the oracle
        ref = []
        for i in range(L.n_layers):
            fill_host_block(L, i, P.arrays[i], "fault", 2)
            ref.append(P.arrays[i].copy())
        hp, ohp = lst.adamw_hparams(step=2), oracle.hparams(step=2)
        lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), hp, 60_000)
        for i in range(L.n_layers):
            oracle_step(L, ref[i], i, ohp)
            assert np.array_equal(P.arrays[i], ref[i])
    finally:
        P.free()


def test_never_observed_completion_times_out():
    L = _small()
    P = PinnedBlocks(L)
    try:
        b0, b1 = _bufs(L)
        lst.lst_test_inject(2, 0)
        t0 = time.time()
        with pytest.raises(lst.LstError) as e:
            lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), lst.adamw_hparams(), 300)
        dt = time.time() - t0
        assert e.value.status == lst.LST_ERR_TIMEOUT
        assert 0.25 <= dt < 30
        lst.lst_test_inject(0, 0)
        lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), lst.adamw_hparams(), 60_000)
    finally:
        P.free()


# ---- zero-copy: the kernel works on the pinned host blocks over the link ----
def _zero_copy_vs_device(specs, fmt, workload, t, steps):
    L = Layout(specs, fmt)
    P = PinnedBlocks(L)
    try:
        for i in range(L.n_layers):
            fill_host_block(L, i, P.arrays[i], workload, t)
        dev = [torch.from_numpy(P.arrays[i].copy()).cuda() for i in range(L.n_layers)]
        ref = [P.arrays[i].copy() for i in range(L.n_layers)]
        s = torch.cuda.current_stream().cuda_stream
        for k in range(steps):
            hp, ohp = hparams_for(workload, t + k)
            lst.lst_adamw_step(L.handle, [d.data_ptr() for d in dev], hp, s)
            lst.lst_zero_copy_step(L.handle, P.ptrs, hp, s)
            torch.cuda.synchronize()
            for i in range(L.n_layers):
                oracle_step(L, ref[i], i, ohp)
        for i in range(L.n_layers):
            assert np.array_equal(P.arrays[i], dev[i].cpu().numpy()), f"block {i}: zero-copy differs"
            compare(fmt, L.numpy_views(i, P.arrays[i]), L.numpy_views(i, ref[i]))
    finally:
        P.free()


@pytest.mark.parametrize("fmt,workload", FMTS)
def test_zero_copy_bit_identical(fmt, workload):
    _zero_copy_vs_device(_three_tinyllama_layers(), fmt, workload, 10, steps=2)


def test_zero_copy_lora_many_blocks():
    _zero_copy_vs_device(shapes.tinyllama_lora(), "L16F", "tinyllama_lora_l16f", 1, steps=2)


def test_zero_copy_rejects_pageable_and_device_memory():
    L = _small()
    pageable = [np.zeros(L.block_bytes(i) + 8192, np.uint8) for i in range(L.n_layers)]
    ptrs = [(a.ctypes.data + 4095) // 4096 * 4096 for a in pageable]
    with pytest.raises(lst.LstError) as e:
        lst.lst_zero_copy_step(L.handle, ptrs, lst.adamw_hparams(), 0)
    assert e.value.status == lst.LST_ERR_NOT_PINNED
    d = [torch.empty(L.block_bytes(i), dtype=torch.uint8, device="cuda") for i in range(L.n_layers)]
    with pytest.raises(lst.LstError) as e:
        lst.lst_zero_copy_step(L.handle, [x.data_ptr() for x in d], lst.adamw_hparams(), 0)
    assert e.value.status == lst.LST_ERR_NOT_PINNED


# ---- gradients already on the device: only the state crosses the link inbound ----
@pytest.mark.parametrize("fmt,workload", FMTS)
@pytest.mark.parametrize("chunk", [0, 1 << 20])
def test_stream_devgrad_bit_identical(fmt, workload, chunk):
    L = Layout(_three_tinyllama_layers(), fmt)
    L.set_stream_chunk(chunk)
    P = PinnedBlocks(L)
    try:
        for i in range(L.n_layers):
            fill_host_block(L, i, P.arrays[i], workload, 10)
        dev = [torch.from_numpy(P.arrays[i].copy()).cuda() for i in range(L.n_layers)]
        grads = [torch.from_numpy(L.numpy_views(i, P.arrays[i])["G"].copy().view(np.uint8)).cuda()
                 for i in range(L.n_layers)]
        # the host G segments now hold something else: they must be neither read nor written
        poison = []
        for i in range(L.n_layers):
            g = L.numpy_views(i, P.arrays[i])["G"].view(np.uint8)
            g[:] = 0x7F
            poison.append(g.copy())
        b0, b1 = _bufs(L)
        for k in range(2):
            hp, _ = hparams_for(workload, 10 + k)
            lst.lst_adamw_step(L.handle, [d.data_ptr() for d in dev], hp, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            lst.lst_stream_step_devgrad(L.handle, P.ptrs, [g.data_ptr() for g in grads], b0.data_ptr(),
                                        b1.data_ptr(), hp, None, 600_000)
        for i in range(L.n_layers):
            got, exp = L.numpy_views(i, P.arrays[i]), L.numpy_views(i, dev[i].cpu().numpy())
            for f in got:
                if f == "G":
                    assert np.array_equal(got[f].view(np.uint8), poison[i])
                else:
                    assert np.array_equal(got[f].view(np.uint8), exp[f].view(np.uint8)), (i, f)
    finally:
        P.free()


def test_stream_devgrad_validation():
    L = _small()
    P = PinnedBlocks(L)
    try:
        b0, b1 = _bufs(L)
        with pytest.raises(lst.LstError) as e:
            lst.lst_stream_step_devgrad(L.handle, P.ptrs, [0] * L.n_layers, b0.data_ptr(), b1.data_ptr(),
                                        lst.adamw_hparams(), None, 10_000)
        assert e.value.status == lst.LST_ERR_INVALID_ARG
        g = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
        with pytest.raises(lst.LstError) as e:
            lst.lst_stream_step_devgrad(L.handle, P.ptrs, [g.data_ptr() + 8] * L.n_layers, b0.data_ptr(),
                                        b1.data_ptr(), lst.adamw_hparams(), None, 10_000)
        assert e.value.status == lst.LST_ERR_ALIGNMENT
    finally:
        P.free()


@pytest.mark.slow
def test_stream_llama7b_full_bit_identical_to_device():
    """LLaMA-7B, 12 B/param, 34 blocks (80.9 GB): the same step device-resident
    and streamed from pinned host memory give the same bytes everywhere."""
    workload, fmt = "llama7b_l12", "L12"
    L = Layout(shapes.llama7b(), fmt)
    P = PinnedBlocks(L)
    try:
        for i in range(L.n_layers):
            fill_host_block(L, i, P.arrays[i], workload, 10)
        dev = []
        for i in range(L.n_layers):
            d = torch.empty(L.block_bytes(i), dtype=torch.uint8, device="cuda")
            d.copy_(torch.from_numpy(P.arrays[i]))
            dev.append(d)
        hp, _ = hparams_for(workload, 10)
        lst.lst_adamw_step(L.handle, [d.data_ptr() for d in dev], hp, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        b0, b1 = _bufs(L)
        lst.lst_stream_step(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), hp, 600_000)
        for i in range(L.n_layers):
            assert torch.equal(dev[i], torch.from_numpy(P.arrays[i]).cuda()), f"block {i}"
    finally:
        P.free()
