"""Per-block options on GB300: step counters, locked blocks, sum of g^2.

Progressive layer locking ("Training 70B Models on Consumer Hardware",
section "Progressive Layer Locking") needs, per layer, its own step counter
(exact bias correction), a way to leave a locked layer untouched (no update,
no I/O) and the gradient magnitude that decides the lock. Checked: per-block
t equals separate single-block calls bit for bit and the oracle; locked
blocks are bit-untouched; sum(g^2) per block within 1e-6 relative of the
oracle's fp64 sum (fp32 partial sums of 8 squares: at most 7 roundings of a
nonnegative sum, 7 * 2^-24 < 5e-7) and deterministic across calls.
"""

import numpy as np
import pytest

import oracle
from optimizer_update_gb300 import Layout, lst
from synth import shapes

from gpu_util import (PinnedBlocks, compare, fill_host_block, gather_device, gathered_inputs, hparams_for,
                      oracle_step, sample_indices)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GSQ_REL = 1e-6


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield
    torch.cuda.synchronize()


def _specs():
    s = [(n, sh, l - 1) for (n, sh, l) in shapes.tinyllama_full() if l in (1, 2)]
    return s + [("odd", (4097,), 2), ("tiny", (9,), 3), ("lora_A", (8, 2048), 4), ("lora_B", (2048, 8), 4)]


def _setup(fmt, workload, t=10):
    L = Layout(_specs(), fmt)
    hosts = [np.empty(L.block_bytes(i), np.uint8) for i in range(L.n_layers)]
    for i in range(L.n_layers):
        fill_host_block(L, i, hosts[i], workload, t)
    return L, hosts


def _ws():
    return torch.empty(lst.lst_workspace_bytes(), dtype=torch.uint8, device="cuda")


FMTS = [("L12", "tinyllama_layer_l12"), ("L16M", "tinyllama_full_l16m"), ("L16F", "tinyllama_lora_l16f")]


@pytest.mark.parametrize("fmt,workload", FMTS)
def test_per_block_steps_skip_and_grad_sq(fmt, workload):
    L, hosts = _setup(fmt, workload)
    steps = [1, 5, 10, 3, 1000][: L.n_layers]
    skip = [0, 0, 1, 0, 0][: L.n_layers]
    dev = [torch.from_numpy(h).cuda() for h in hosts]
    gsq = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
    ws = _ws()
    hp, _ = hparams_for(workload, 7)
    opts = lst.step_options(block_steps=steps, skip=skip, grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
    lst.lst_adamw_step_ex(L.handle, [d.data_ptr() for d in dev], hp, opts, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    # the same blocks one at a time through the plain call, each with its own t
    single = []
    for i in range(L.n_layers):
        Li = Layout([(n, sh, 0) for (n, sh, l) in _specs() if l == i], fmt)
        d = torch.from_numpy(hosts[i]).cuda()
        if not skip[i]:
            lst.lst_adamw_step(Li.handle, [d.data_ptr()], hparams_for(workload, steps[i])[0],
                               torch.cuda.current_stream().cuda_stream)
        single.append(d)
    torch.cuda.synchronize()
    g = gsq.cpu().numpy()
    for i in range(L.n_layers):
        got = dev[i].cpu().numpy()
        if skip[i]:
            assert np.array_equal(got, hosts[i]), "a locked block must be bit-untouched"
            assert g[i] == -1.0, "a locked block's grad_sq entry is left as it was"
            continue
        assert np.array_equal(got, single[i].cpu().numpy()), f"block {i}: differs from the single-block call"
        exp_g = oracle.grad_sq(L.numpy_views(i, hosts[i])["G"])
        ref = hosts[i].copy()
        oracle_step(L, ref, i, hparams_for(workload, steps[i])[1])
        compare(fmt, L.numpy_views(i, got), L.numpy_views(i, ref))
        assert abs(g[i] - exp_g) <= GSQ_REL * exp_g, (i, g[i], exp_g)


def test_grad_sq_deterministic_and_without_skip():
    fmt, workload = "L12", "tinyllama_layer_l12"
    L, hosts = _setup(fmt, workload)
    ws = _ws()
    out = []
    for rep in range(2):
        dev = [torch.from_numpy(h).cuda() for h in hosts]
        gsq = torch.zeros(L.n_layers, dtype=torch.float64, device="cuda")
        opts = lst.step_options(grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
        lst.lst_adamw_step_ex(L.handle, [d.data_ptr() for d in dev], hparams_for(workload, 4)[0], opts, 0)
        torch.cuda.synchronize()
        out.append(gsq.cpu().numpy())
        # without per-block steps or skip, the result equals the plain step bit for bit
        plain = [torch.from_numpy(h).cuda() for h in hosts]
        lst.lst_adamw_step(L.handle, [d.data_ptr() for d in plain], hparams_for(workload, 4)[0], 0)
        torch.cuda.synchronize()
        for a, b in zip(dev, plain):
            assert torch.equal(a, b)
    assert np.array_equal(out[0].view(np.uint64), out[1].view(np.uint64))


def test_grad_sq_lora_full_size():
    fmt, workload = "L16F", "tinyllama_lora_l16f"
    L = Layout(shapes.tinyllama_lora(), fmt)
    hosts = [np.empty(L.block_bytes(i), np.uint8) for i in range(L.n_layers)]
    for i in range(L.n_layers):
        fill_host_block(L, i, hosts[i], workload, 10)
    dev = [torch.from_numpy(h).cuda() for h in hosts]
    gsq = torch.zeros(L.n_layers, dtype=torch.float64, device="cuda")
    ws = _ws()
    opts = lst.step_options(grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
    lst.lst_adamw_step_ex(L.handle, [d.data_ptr() for d in dev], hparams_for(workload, 10)[0], opts, 0)
    torch.cuda.synchronize()
    g = gsq.cpu().numpy()
    for i in range(L.n_layers):
        exp_g = oracle.grad_sq(L.numpy_views(i, hosts[i])["G"])
        assert abs(g[i] - exp_g) <= GSQ_REL * exp_g


@pytest.mark.parametrize("fmt,workload", FMTS)
def test_small_launches_many_ragged_blocks(fmt, workload):
    """130 small blocks of ragged sizes (two launches of the cross-run
    small-launch kernel): per-block steps, every 11th block locked, sum of g^2
    for the rest; each block against the oracle, and the sums bit-identical on
    a second call."""
    specs = [(f"t{i}", ((i * 7919) % 6000 + 1,), i) for i in range(130)]
    specs += [(f"u{i}", (3, (i * 31) % 700 + 1), i) for i in range(0, 130, 3)]
    L = Layout(specs, fmt)
    hosts = [np.empty(L.block_bytes(i), np.uint8) for i in range(L.n_layers)]
    for i in range(L.n_layers):
        fill_host_block(L, i, hosts[i], workload, 10)
    steps = [1 + (i * 13) % 50 for i in range(L.n_layers)]
    skip = [1 if i % 11 == 4 else 0 for i in range(L.n_layers)]
    ws = _ws()
    sums = []
    for rep in range(2):
        dev = [torch.from_numpy(h).cuda() for h in hosts]
        gsq = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
        opts = lst.step_options(block_steps=steps, skip=skip, grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
        lst.lst_adamw_step_ex(L.handle, [d.data_ptr() for d in dev], hparams_for(workload, 3)[0], opts,
                              torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        sums.append(gsq.cpu().numpy())
    g = sums[0]
    assert np.array_equal(sums[0].view(np.uint64), sums[1].view(np.uint64))
    for i in range(L.n_layers):
        got = dev[i].cpu().numpy()
        if skip[i]:
            assert np.array_equal(got, hosts[i]) and g[i] == -1.0
            continue
        ref = hosts[i].copy()
        oracle_step(L, ref, i, hparams_for(workload, steps[i])[1], threads=1)
        compare(fmt, L.numpy_views(i, got), L.numpy_views(i, ref))
        exp_g = oracle.grad_sq(L.numpy_views(i, hosts[i])["G"])
        assert abs(g[i] - exp_g) <= GSQ_REL * exp_g, (i, g[i], exp_g)


@pytest.mark.slow
def test_full_size_mixed_layout_sampled():
    """The whole TinyLlama-1.1B mixed-layout state (17.6 GB) in one extended
    launch, as the bench times it (three waves of CTAs): per-block steps
    t + (block mod 4), block 5 locked, sums of g^2 for the rest. Sampled
    elements of every block against the oracle at that block's own step, the
    locked block bit-untouched, every sum against the oracle's."""
    fmt, workload, t = "L16M", "tinyllama_full_l16m", 10
    L = Layout(shapes.tinyllama_full(), fmt)
    host = np.empty(L.max_block_bytes, np.uint8)
    blocks, exp_g = [], []
    for i in range(L.n_layers):
        n = L.block_bytes(i)
        fill_host_block(L, i, host[:n], workload, t)
        exp_g.append(oracle.grad_sq(L.numpy_views(i, host[:n])["G"]))
        b = torch.empty(n, dtype=torch.uint8, device="cuda")
        b.copy_(torch.from_numpy(host[:n]))
        blocks.append(b)
    locked = 5
    before = blocks[locked].clone()
    steps = [t + i % 4 for i in range(L.n_layers)]
    skip = [1 if i == locked else 0 for i in range(L.n_layers)]
    gsq = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
    ws = _ws()
    opts = lst.step_options(block_steps=steps, skip=skip, grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
    lst.lst_adamw_step_ex(L.handle, [b.data_ptr() for b in blocks], hparams_for(workload, t)[0], opts,
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(blocks[locked], before)
    g = gsq.cpu().numpy()
    rng = np.random.default_rng(7)
    checked = 0
    for i in range(L.n_layers):
        if i == locked:
            assert g[i] == -1.0
            continue
        assert abs(g[i] - exp_g[i]) <= GSQ_REL * exp_g[i], (i, g[i], exp_g[i])
        idx = sample_indices(L.padded(i), L.spans(i), rng, n_random=4096)
        inp = gathered_inputs(L, i, workload, t, idx)
        oracle.step(fmt, inp, hparams_for(workload, steps[i])[1])
        compare(fmt, gather_device(L.torch_views(i, blocks[i]), idx), inp)
        checked += idx.size
    assert checked > 50_000


@pytest.mark.parametrize("fmt,workload", FMTS)
@pytest.mark.parametrize("chunk", [0, 1 << 20])
def test_stream_step_ex(fmt, workload, chunk):
    L, hosts = _setup(fmt, workload)
    L.set_stream_chunk(chunk)
    steps = [2, 9, 4, 1, 30][: L.n_layers]
    skip = [0, 1, 0, 0, 0][: L.n_layers]
    P = PinnedBlocks(L)
    try:
        for i in range(L.n_layers):
            P.arrays[i][:] = hosts[i]
        b0 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        b1 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        gsq = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
        ws = _ws()
        hp, _ = hparams_for(workload, 1)
        opts = lst.step_options(block_steps=steps, skip=skip, grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
        lst.lst_stream_step_ex(L.handle, P.ptrs, b0.data_ptr(), b1.data_ptr(), hp, opts, 600_000)
        # device-resident reference with the same options
        dev = [torch.from_numpy(h).cuda() for h in hosts]
        lst.lst_adamw_step_ex(L.handle, [d.data_ptr() for d in dev], hp,
                              lst.step_options(block_steps=steps, skip=skip), 0)
        torch.cuda.synchronize()
        g = gsq.cpu().numpy()
        for i in range(L.n_layers):
            assert np.array_equal(P.arrays[i], dev[i].cpu().numpy()), f"block {i}"
            if skip[i]:
                assert np.array_equal(P.arrays[i], hosts[i]) and g[i] == -1.0
                continue
            exp_g = oracle.grad_sq(L.numpy_views(i, hosts[i])["G"])
            assert abs(g[i] - exp_g) <= GSQ_REL * exp_g, (i, g[i], exp_g)
    finally:
        P.free()
