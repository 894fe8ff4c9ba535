"""Device-resident step vs the oracle, element by element (GB300).

Small and medium workloads are compared in full; the full-size workloads
(TinyLlama-1.1B mixed, LLaMA-7B) on sampled elements that the oracle computes
one by one from the generator's inputs at those indices. Tolerances: fp32
fields within 1e-6 relative (+1e-30 absolute), bf16 weights within one bf16
ulp of the oracle's round-to-nearest-even result; the kernel is also expected
to be bit-exact (same fp32 operation order, IEEE division and square root).
"""

import numpy as np
import pytest

import oracle
from optimizer_update_gb300 import Layout, lst
from synth import shapes

from gpu_util import (FIELD_DT, compare, device_blocks, fill_host_block, gather_device, gathered_inputs,
                      guards_intact, hparams_for, oracle_step, sample_indices)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _run_full(specs, fmt, workload, t, sgd=False, guard=4096, hp_override=None):
    """Fill, step on the device, step the oracle, compare every field of every block."""
    L = Layout(specs, fmt)
    hosts = [np.empty(L.block_bytes(i), np.uint8) for i in range(L.n_layers)]
    for i in range(L.n_layers):
        fill_host_block(L, i, hosts[i], workload, t)
    blocks, backing = device_blocks(L, guard=guard)
    for i in range(L.n_layers):
        blocks[i].copy_(torch.from_numpy(hosts[i]))
    hp, ohp = hparams_for(workload, t)
    if hp_override:
        for k, v in hp_override.items():
            setattr(hp, k, v)
            setattr(ohp, k, v)
    ptrs = [b.data_ptr() for b in blocks]
    if sgd:
        lst.lst_sgd_step(L.handle, ptrs, hp.lr, _stream())
    else:
        lst.lst_adamw_step(L.handle, ptrs, hp, _stream())
    torch.cuda.synchronize()
    stats = []
    for i in range(L.n_layers):
        before_g = L.numpy_views(i, hosts[i])["G"].copy()
        oracle_step(L, hosts[i], i, ohp, sgd=sgd)
        got = L.numpy_views(i, blocks[i].cpu().numpy())
        exp = L.numpy_views(i, hosts[i])
        fields = ("W",) if (sgd and fmt != "L16M") else (("MASTER", "W") if sgd else None)
        s = compare(fmt, got, exp, fields)
        assert np.array_equal(got["G"], before_g), "gradient must be read-only"
        if sgd:  # moments untouched
            assert np.array_equal(got["M"].view(np.uint32), exp["M"].view(np.uint32))
            assert np.array_equal(got["V"].view(np.uint32), exp["V"].view(np.uint32))
        stats.append(s)
    if guard:
        assert guards_intact(backing, L, guard), "write outside a block"
    return L, stats


def _assert_bit_exact(stats):
    for s in stats:
        for f, d in s.items():
            assert d["bit_exact"] == d["n"], f"{f}: {d['n'] - d['bit_exact']} elements not bit-exact"


# ---- one TinyLlama-1.1B decoder layer, 12 B/param, t = 1 (m = v = 0) and t = 10
@pytest.mark.parametrize("t", [1, 10])
def test_tinyllama_layer_l12_full(t):
    _, stats = _run_full(shapes.tinyllama_layer(), "L12", "tinyllama_layer_l12", t)
    _assert_bit_exact(stats)


# ---- TinyLlama LoRA r=8 adapters (308 tensors, 22 blocks), fp32, multi-block launch
@pytest.mark.parametrize("t", [1, 10])
def test_tinyllama_lora_l16f_full(t):
    # the frozen bf16 base (1.1B parameters) is resident but never passed to
    # the library: it must come through bit-untouched
    base = torch.randint(-32768, 32767, (1_100_048_384,), dtype=torch.int16, device="cuda")
    ck = int(base.view(torch.int32)[: base.numel() // 2].sum(dtype=torch.int64))
    _, stats = _run_full(shapes.tinyllama_lora(), "L16F", "tinyllama_lora_l16f", t)
    _assert_bit_exact(stats)
    assert int(base.view(torch.int32)[: base.numel() // 2].sum(dtype=torch.int64)) == ck
    del base


# ---- odd sizes: 1, 7, 9, 4097 elements, a scalar, an empty tensor, several blocks
EDGE = [("scalar", (), 0), ("one", (1,), 0), ("seven", (7,), 0), ("nine", (9,), 1),
        ("tail", (4097,), 1), ("empty", (0, 3), 2), ("x", (5, 3), 2), ("big", (70_001,), 3)]


@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
@pytest.mark.parametrize("sgd", [False, True])
def test_edge_shapes(fmt, sgd):
    _, stats = _run_full(EDGE, fmt, "edge", 7, sgd=sgd)
    _assert_bit_exact(stats)


def test_mixed_layout_three_layers():
    specs = [s for s in shapes.tinyllama_full() if s[2] in (1, 2, 3)]
    specs = [(n, sh, l - 1) for (n, sh, l) in specs]
    _, stats = _run_full(specs, "L16M", "tinyllama_full_l16m", 10)
    _assert_bit_exact(stats)


@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
def test_lr_zero_keeps_weights(fmt):
    L = Layout(shapes.tinyllama_layer()[:3], fmt)
    host = np.empty(L.block_bytes(0), np.uint8)
    fill_host_block(L, 0, host, "lr0", 5)
    blk = torch.from_numpy(host).cuda()
    hp, _ = hparams_for("lr0", 5)
    hp.lr = 0.0
    lst.lst_adamw_step(L.handle, [blk.data_ptr()], hp, _stream())
    torch.cuda.synchronize()
    got, before = L.numpy_views(0, blk.cpu().numpy()), L.numpy_views(0, host)
    wf = "MASTER" if fmt == "L16M" else "W"
    # the input weights hold no -0.0 (lattice draws): w*1 - 0*u is w bit for bit
    assert np.array_equal(got[wf].view(np.uint8), before[wf].view(np.uint8))
    assert not np.array_equal(got["M"], before["M"]) and not np.array_equal(got["V"], before["V"])


def test_more_blocks_than_one_launch_holds():
    # 300 small blocks: the run table is split over several launches
    specs = [(f"t{i}", (1000 + 37 * i,), i) for i in range(300)]
    _, stats = _run_full(specs, "L12", "many", 3)
    _assert_bit_exact(stats)


def test_padding_stays_zero():
    L = Layout([("a", (5,), 0), ("b", (3000,), 0)], "L16M")
    host = np.zeros(L.block_bytes(0), np.uint8)
    fill_host_block(L, 0, host, "pad", 4)
    blk = torch.from_numpy(host).cuda()
    lst.lst_adamw_step(L.handle, [blk.data_ptr()], hparams_for("pad", 4)[0], _stream())
    torch.cuda.synchronize()
    v = L.numpy_views(0, blk.cpu().numpy())
    used = np.zeros(L.padded(0), bool)
    for (_, off, n) in L.spans(0):
        used[off:off + n] = True
    for f, arr in v.items():
        assert not np.any(arr[~used]), f


# ---- full sizes, sampled (the launch configuration the bench times: one
# multi-block launch over every block of the model)
def _full_size_sampled(specs, fmt, workload, t, seed_rng, sgd=False):
    L = Layout(specs, fmt)
    host = np.empty(L.max_block_bytes, np.uint8)
    blocks = []
    for i in range(L.n_layers):
        n = L.block_bytes(i)
        fill_host_block(L, i, host[:n], workload, t)
        b = torch.empty(n, dtype=torch.uint8, device="cuda")
        b.copy_(torch.from_numpy(host[:n]))
        blocks.append(b)
    hp, ohp = hparams_for(workload, t)
    if sgd:
        lst.lst_sgd_step(L.handle, [b.data_ptr() for b in blocks], hp.lr, _stream())
    else:
        lst.lst_adamw_step(L.handle, [b.data_ptr() for b in blocks], hp, _stream())
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed_rng)
    checked = 0
    for i in range(L.n_layers):
        idx = sample_indices(L.padded(i), L.spans(i), rng)
        inp = gathered_inputs(L, i, workload, t, idx)
        before = {f: a.copy() for f, a in inp.items()}
        oracle.step(fmt, inp, ohp, sgd=sgd)
        got = gather_device(L.torch_views(i, blocks[i]), idx)
        fields = (("MASTER", "W") if fmt == "L16M" else ("W",)) if sgd else None
        s = compare(fmt, got, inp, fields)
        _assert_bit_exact([s])
        if sgd:  # the moments are neither read nor written
            for f in ("M", "V"):
                assert np.array_equal(got[f].view(np.uint32), before[f].view(np.uint32)), f
        checked += idx.size
    del blocks
    return checked


@pytest.mark.slow
def test_tinyllama_full_l16m_sampled():
    assert _full_size_sampled(shapes.tinyllama_full(), "L16M", "tinyllama_full_l16m", 10, 1) > 100_000


@pytest.mark.slow
def test_llama7b_l12_sampled():
    assert _full_size_sampled(shapes.llama7b(), "L12", "llama7b_l12", 10, 2) > 100_000


# ---- the SGD form through the large-launch kernels (the launches the bench
# times): three TinyLlama-1.1B layers per layout in one launch, every element
# of every block against the oracle, bit for bit (one and two waves of CTAs)
@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
def test_sgd_three_layers_large_launch_full(fmt):
    specs = [(n, sh, l - 1) for (n, sh, l) in shapes.tinyllama_full() if l in (1, 2, 3)]
    L, stats = _run_full(specs, fmt, "tinyllama_full_l16m" if fmt == "L16M" else "sgd_three_layers", 4, sgd=True)
    alg = 22 if fmt == "L12" else 28
    assert L.n_params * alg > (256 << 20)  # above the small-launch threshold
    _assert_bit_exact(stats)


# ... and over the whole TinyLlama-1.1B state (more than 8 GB per launch: the
# 16 B layouts' three-wave grid), sampled
@pytest.mark.slow
@pytest.mark.parametrize("fmt", ["L16M", "L16F"])
def test_sgd_tinyllama_full_sampled(fmt):
    assert _full_size_sampled(shapes.tinyllama_full(), fmt, "tinyllama_full_l16m", 6, 3, sgd=True) > 100_000


@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
@pytest.mark.parametrize("eps", [1e-8, 0.0])
def test_zeros_signed_zeros_and_tiny_values_bit_exact(fmt, eps):
    """Exact zeros (in g, m, v, w), negative zeros and subnormal-range values:
    the cases in which the kernel substitutes known IEEE results for the
    division and square root must still match the oracle bit for bit (with
    eps = 0 a zero moment gives 0/0 = NaN on both sides)."""
    n = 4096 * 8
    L = Layout([("x", (n,), 0)], fmt)
    host = np.zeros(L.block_bytes(0), np.uint8)
    v = L.numpy_views(0, host)
    rng = np.random.default_rng(77)
    kinds = rng.integers(0, 6, n)
    def pick(scale):
        x = (rng.standard_normal(n) * scale).astype(np.float32)
        x[kinds == 0] = 0.0
        x[kinds == 1] = -0.0
        x[kinds == 2] *= np.float32(1e-36)          # subnormal-range products
        return x
    g32, m32 = pick(1e-3), pick(1e-4)
    v32 = np.abs(pick(1e-6)).astype(np.float32)
    v32[kinds == 1] = 0.0
    w32 = pick(0.02)
    if fmt == "L16F":
        v["G"][:] = g32
        v["W"][:] = w32
    else:
        v["G"][:] = oracle.bf16_from_f32(g32)
        if fmt == "L12":
            v["W"][:] = oracle.bf16_from_f32(w32)
        else:
            v["MASTER"][:] = w32
    v["M"][:] = m32
    v["V"][:] = v32
    blk = torch.from_numpy(host).cuda()
    hp_kw = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=eps, weight_decay=0.01, step=3)
    lst.lst_adamw_step(L.handle, [blk.data_ptr()], lst.adamw_hparams(**hp_kw), _stream())
    torch.cuda.synchronize()
    oracle.step(fmt, L.numpy_views(0, host), oracle.hparams(**hp_kw))
    got, exp = L.numpy_views(0, blk.cpu().numpy()), L.numpy_views(0, host)
    for f in got:
        if f == "G":
            continue
        if got[f].dtype == np.float32:
            gn, en = np.isnan(got[f]), np.isnan(exp[f])
            assert np.array_equal(gn, en), f
            assert np.array_equal(got[f][~gn].view(np.uint32), exp[f][~en].view(np.uint32)), f
        else:
            gf, ef = oracle.f32_from_bf16(got[f]), oracle.f32_from_bf16(exp[f])
            assert np.array_equal(np.isnan(gf), np.isnan(ef)), f
            ok = ~np.isnan(ef)
            assert np.array_equal(got[f][ok], exp[f][ok]), f


# ---- large launches with ragged blocks: blocks of 1, 9, 4097 and 70,001
# elements (segments that end inside a warp's 256-element task span, padded)
# in one launch with full TinyLlama-1.1B layers, above the small-launch
# threshold: every element against the oracle, bit for bit.
@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
@pytest.mark.parametrize("sgd", [False, True])
def test_large_launch_ragged_blocks_full(fmt, sgd):
    specs = [(n, sh, 0) for (n, sh, l) in shapes.tinyllama_full() if l == 1]
    specs += [("one", (1,), 1), ("nine", (9,), 2), ("odd", (4097,), 2), ("big_odd", (70001,), 3)]
    specs += [(n, sh, 4) for (n, sh, l) in shapes.tinyllama_full() if l == 2]
    specs += [("tail", (2048 * 3 + 256,), 5)]
    L, stats = _run_full(specs, fmt, "tinyllama_full_l16m" if fmt == "L16M" else "ragged_large", 7, sgd=sgd)
    assert L.n_params * (22 if fmt == "L12" else 28) > (256 << 20)  # one large launch
    _assert_bit_exact(stats)
