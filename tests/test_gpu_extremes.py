"""Extreme and non-finite inputs through every update kernel, against the oracle (GB300).

"The Math" ("Training 70B Models on Consumer Hardware (If You're Willing to
Wait)") defines the update for every input, and IEEE arithmetic fixes its
result for every operand: infinities, NaN, gradients whose square overflows
fp32 (|g| >= 2^64, so v becomes +inf), negative or infinite second moments,
a huge step count (bias corrections of exactly 1), betas of 0 (m = g,
v = g^2), lr * wd = 1 (the decay factor 0) and eps of 0 or below 0 (a zero
or negative denominator). The generator's draws are bounded, so these inputs
are written here directly.

Every case runs through the small-launch kernel (one 64 Ki-element block)
and the large-launch kernel (two blocks, 16 Mi elements, over the 256 MB
threshold), plain (lst_adamw_step) and with per-block options
(lst_adamw_step_ex: its own kernels), and the SGD form. Results are compared
with the oracle bit for bit, except that NaN compares equal to NaN whatever
its payload (the device writes the canonical quiet NaN; the host's arithmetic
passes an input NaN's payload on).
"""

import numpy as np
import pytest

import oracle
from optimizer_update_gb300 import Layout, lst

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


INF = np.float32(np.inf)
BIG_G = np.float32(2.0 ** 64)        # g*g = 2^128 overflows fp32: v becomes +inf
HUGE_G = np.float32(2.0 ** 100)
BF16_MAX = np.float32(3.3895313892515355e38)
TINY = np.float32(1e-40)             # subnormal in fp32 (and bf16)

SPECIAL = {
    "G": [INF, -INF, np.nan, BIG_G, -BIG_G, HUGE_G, -HUGE_G, BF16_MAX, -BF16_MAX, 0.0, -0.0, TINY, -TINY],
    "M": [INF, -INF, np.nan, 0.0, -0.0, np.float32(1e38), np.float32(-1e38), TINY],
    "V": [INF, np.nan, 0.0, -0.0, np.float32(-1e-6), np.float32(1e38), TINY, np.float32(-INF)],
    "W": [INF, -INF, np.nan, 0.0, -0.0, BF16_MAX, -BF16_MAX, TINY, np.float32(1e30)],
}
SCALE = {"G": 1e-3, "M": 1e-4, "V": 1e-3, "W": 0.02}

HPARAMS = {
    "ordinary": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=3),
    "t_1e6": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=10 ** 6),
    "betas_0": dict(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8, weight_decay=0.01, step=2),
    "lr_wd_1": dict(lr=0.5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=2.0, step=5),
    "eps_0": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=0.0, weight_decay=0.0, step=1),
    "eps_neg": dict(lr=1e-3, beta1=0.5, beta2=0.75, eps=-1e-3, weight_decay=0.1, step=7),
}

SMALL = 65536              # one block: lst_update_small_kernel
LARGE = 8 * 1024 * 1024    # per block, two blocks: above the 256 MB small-launch threshold


def _values(rng, name, n):
    """Ordinary draws with about one element in three replaced by a special
    value of the field (v's ordinary draws are squares)."""
    x = (rng.standard_normal(n) * SCALE[name]).astype(np.float32)
    if name == "V":
        x = x * x
    sp = np.array(SPECIAL[name], dtype=np.float32)
    pick = rng.integers(0, 3 * sp.size, n)
    sel = pick < sp.size
    x[sel] = sp[pick[sel]]
    return x


def _fill(L, host, i, fmt, rng):
    v = L.numpy_views(i, host)
    n = L.block(i)[1]
    g, m, vv, w = (_values(rng, k, n) for k in ("G", "M", "V", "W"))
    if fmt == "L16F":
        v["G"][:n], v["W"][:n] = g, w
    else:
        v["G"][:n] = oracle.bf16_from_f32(g)
        if fmt == "L12":
            v["W"][:n] = oracle.bf16_from_f32(w)
        else:
            v["MASTER"][:n] = w
    v["M"][:n], v["V"][:n] = m, vv


OUTPUTS = {"L12": ("W", "M", "V"), "L16M": ("MASTER", "M", "V", "W"), "L16F": ("W", "M", "V")}


def _case(fmt, n_per_block, n_blocks, hp_kw, seed, kernel):
    L = Layout([(f"t{i}", (n_per_block - 5 * i,), i) for i in range(n_blocks)], fmt)
    rng = np.random.default_rng(seed)
    hosts = []
    for i in range(L.n_layers):
        h = np.zeros(L.block_bytes(i), np.uint8)
        _fill(L, h, i, fmt, rng)
        hosts.append(h)
    dev = [torch.from_numpy(h).cuda() for h in hosts]
    ptrs = [d.data_ptr() for d in dev]
    stream = torch.cuda.current_stream().cuda_stream
    sgd = kernel == "sgd"
    gsq = None
    if kernel == "plain":
        lst.lst_adamw_step(L.handle, ptrs, lst.adamw_hparams(**hp_kw), stream)
    elif kernel == "sgd":
        lst.lst_sgd_step(L.handle, ptrs, hp_kw["lr"], stream)
    else:  # per-block options: every block at the same step, sums of g^2 on
        gsq = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
        ws = torch.empty(lst.lst_workspace_bytes(), dtype=torch.uint8, device="cuda")
        opts = lst.step_options(block_steps=[hp_kw["step"]] * L.n_layers, grad_sq=gsq.data_ptr(),
                                workspace=ws.data_ptr())
        lst.lst_adamw_step_ex(L.handle, ptrs, lst.adamw_hparams(**hp_kw), opts, stream)
    torch.cuda.synchronize()
    for i in range(L.n_layers):
        exp = L.numpy_views(i, hosts[i])
        g_in = exp["G"].copy()
        oracle.step(fmt, exp, oracle.hparams(**hp_kw), sgd=sgd, threads=8)
        got = L.numpy_views(i, dev[i].cpu().numpy())
        assert np.array_equal(got["G"].view(np.uint8), g_in.view(np.uint8)), "gradient must be read-only"
        if sgd:
            for f in ("M", "V"):
                assert np.array_equal(got[f].view(np.uint32), exp[f].view(np.uint32)), f
            _same_fields(got, exp, ("MASTER", "W") if fmt == "L16M" else ("W",))
        else:
            _same_fields(got, exp, OUTPUTS[fmt])
        if gsq is not None:
            gv = g_in if fmt == "L16F" else oracle.f32_from_bf16(g_in)
            s = float(gsq[i].item())
            if np.isnan(gv).any():
                assert np.isnan(s), (i, s)
            else:  # +inf from an infinite g, or from a square beyond fp32's range
                assert s == np.inf, (i, s)


def _same_fields(got, exp, fields):
    """The given fields bit for bit; NaN equal to NaN (bf16 fields as bit
    patterns)."""
    for f in fields:
        a, b = got[f], exp[f]
        if a.dtype == np.float32:
            an, bn, ai, bi = np.isnan(a), np.isnan(b), a.view(np.uint32), b.view(np.uint32)
        else:
            an, bn, ai, bi = (a & 0x7FFF) > 0x7F80, (b & 0x7FFF) > 0x7F80, a, b
        assert np.array_equal(an, bn), f"{f}: NaN at different elements ({int((an != bn).sum())})"
        diff = np.nonzero(ai[~an] != bi[~bn])[0]
        assert diff.size == 0, (f"{f}: {diff.size} elements differ; first: got {a[~an][diff[0]]!r} "
                                f"expected {b[~bn][diff[0]]!r}")


@pytest.mark.parametrize("kernel", ["plain", "options"])
@pytest.mark.parametrize("case", sorted(HPARAMS))
@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
def test_extremes_small_launch(fmt, case, kernel):
    _case(fmt, SMALL, 1, HPARAMS[case], 101, kernel)


@pytest.mark.parametrize("kernel", ["plain", "options"])
@pytest.mark.parametrize("case", ["ordinary", "t_1e6", "betas_0", "lr_wd_1", "eps_neg"])
@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
def test_extremes_large_launch(fmt, case, kernel):
    _case(fmt, LARGE, 2, HPARAMS[case], 202, kernel)


@pytest.mark.parametrize("n,blocks", [(SMALL, 1), (LARGE, 2)])
@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
def test_extremes_sgd(fmt, n, blocks):
    _case(fmt, n, blocks, dict(HPARAMS["ordinary"], lr=0.5), 303, "sgd")
