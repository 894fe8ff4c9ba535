"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test states a fact that follows from the method's definition without
re-evaluating the oracle's own formula: closed forms of the Adam recurrence,
special cases that reduce to plain decay or to an identity, an independent
library conversion, and exact rational arithmetic within a derived rounding
bound. A plausible slip in the oracle (a swapped beta, a dropped term, a wrong
sign, an off-by-one step index, eps under the root, decay after the step, an
index shift) fails at least one of them.
"""

import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import hparams

F32 = np.float32
U = 2.0 ** -24  # unit roundoff of fp32


def _grad_vector(n=257, seed=3):
    rng = np.random.default_rng(seed)
    mag = 10.0 ** rng.uniform(-5, 0, n)           # |g| from 1e-5 to 1: all >> eps = 1e-8
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return (sign * mag).astype(F32)


def _weights(n, seed=4):
    rng = np.random.default_rng(seed)
    return rng.uniform(0.5, 2.0, n).astype(F32) * np.where(rng.random(n) < 0.5, -1, 1).astype(F32)


# ---------------------------------------------------------------------------
# Constant gradient from a zero state: the bias corrections undo the moment
# averaging exactly, so m_t = (1 - b1^t) g, v_t = (1 - b2^t) g^2 and the step
# is lr * g / (|g| + eps) at EVERY t. ("The Math": m_hat = m / (1 - b1^t),
# v_hat = v / (1 - b2^t), W -= lr * m_hat / (sqrt(v_hat) + eps).)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("b1,b2", [(0.9, 0.999), (0.5, 0.75)])
def test_constant_gradient_closed_form_every_step(b1, b2):
    g = _grad_vector()
    n = g.size
    W = _weights(n)
    m = np.zeros(n, F32)
    v = np.zeros(n, F32)
    lr, eps = 1e-3, 1e-8
    gd = g.astype(np.float64)
    # the hyperparameters are fp32: the closed form uses their fp32 values
    B1, B2 = float(F32(b1)), float(F32(b2))
    for t in range(1, 41):
        W_prev = W.astype(np.float64)
        oracle.adamw_l16f(g, W, m, v, hparams(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=0.0, step=t))
        m_exp = (1.0 - B1 ** t) * gd
        v_exp = (1.0 - B2 ** t) * gd * gd
        # t steps of a 3-op recurrence: allow a few ulps per step
        assert np.all(np.abs(m - m_exp) <= 4 * t * U * np.abs(gd) + 1e-45), t
        assert np.all(np.abs(v - v_exp) <= 6 * t * U * gd * gd + 1e-45), t
        step_exp = lr * gd / (np.abs(gd) + eps)
        dW = W.astype(np.float64) - W_prev
        # W is fp32 near 1: one rounding of the weight plus a relative error on the step
        tol = np.spacing(np.abs(W_prev).astype(F32)).astype(np.float64) + 1e-4 * lr
        assert np.all(np.abs(dW + step_exp) <= tol), t


def test_step_one_closed_form_sign_and_magnitude():
    """t = 1 from zero state: m_hat = g, v_hat = g^2, so with wd = 0 the weight
    moves by lr * (1 - eps/|g|) against the sign of g (to first order)."""
    g = _grad_vector(1001, seed=11)
    W = np.zeros(g.size, F32) + F32(0.0)
    W[:] = F32(0.25)
    m = np.zeros(g.size, F32)
    v = np.zeros(g.size, F32)
    lr = 0.125
    oracle.adamw_l16f(g, W, m, v, hparams(lr=lr, eps=1e-8, weight_decay=0.0, step=1))
    gd = g.astype(np.float64)
    # m_hat and v_hat from the stored moments: within a couple of ulps of g, g^2
    B1, B2 = float(F32(0.9)), float(F32(0.999))
    assert np.allclose(m / (1 - B1), gd, rtol=8 * U, atol=0)
    assert np.allclose(v / (1 - B2), gd * gd, rtol=16 * U, atol=0)
    dW = W.astype(np.float64) - 0.25
    assert np.all(np.sign(dW) == -np.sign(gd))
    assert np.allclose(np.abs(dW), lr * np.abs(gd) / (np.abs(gd) + 1e-8), rtol=0, atol=4e-8)


def test_eps_outside_the_root():
    """|g| = eps at t = 1: m_hat/(sqrt(v_hat)+eps) = g/(2 eps) = +-1/2. With eps
    under the root the step would be about 1e-4 instead."""
    eps = 1e-8
    g = np.array([eps, -eps, 2 * eps, -0.5 * eps], F32)
    W = np.zeros(4, F32)
    m = np.zeros(4, F32)
    v = np.zeros(4, F32)
    oracle.adamw_l16f(g, W, m, v, hparams(lr=1.0, eps=eps, weight_decay=0.0, step=1))
    gd = g.astype(np.float64)
    expect = -gd / (np.abs(gd) + eps)            # -0.5, +0.5, -2/3, +1/3
    assert np.allclose(W, expect, rtol=1e-5, atol=0)


def test_two_steps_weighted_average():
    """g1 then g2 from zero: m_hat_2 = (b1 g1 + g2)/(1 + b1) and
    v_hat_2 = (b2 g1^2 + g2^2)/(1 + b2) (geometric weights, bias corrected at t=2)."""
    rng = np.random.default_rng(5)
    n = 513
    g1 = (rng.standard_normal(n) * 1e-2).astype(F32)
    g2 = (rng.standard_normal(n) * 1e-2).astype(F32)
    W = _weights(n)
    m = np.zeros(n, F32)
    v = np.zeros(n, F32)
    b1, b2, lr, eps = float(F32(0.9)), float(F32(0.999)), 1e-3, 1e-8
    oracle.adamw_l16f(g1, W, m, v, hparams(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=0.0, step=1))
    W1 = W.astype(np.float64)
    oracle.adamw_l16f(g2, W, m, v, hparams(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=0.0, step=2))
    a, b = g1.astype(np.float64), g2.astype(np.float64)
    mh = (b1 * a + b) / (1 + b1)
    vh = (b2 * a * a + b * b) / (1 + b2)
    step = lr * mh / (np.sqrt(vh) + eps)
    tol = np.spacing(np.abs(W1).astype(F32)).astype(np.float64) + 1e-4 * np.abs(step) + 1e-12
    assert np.all(np.abs((W.astype(np.float64) - W1) + step) <= tol)


# ---------------------------------------------------------------------------
# Special cases that reduce to simpler maps.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", ["L12", "L16M", "L16F"])
def test_lr_zero_leaves_weights_bit_identical(fmt):
    rng = np.random.default_rng(7)
    n = 4099
    g32 = (rng.standard_normal(n) * 1e-3).astype(F32)
    w32 = (rng.standard_normal(n) * 0.02).astype(F32)
    w32[w32 == 0] = F32(1e-3)  # no signed zeros: -0 - (-0) would become +0
    m0 = (rng.standard_normal(n) * 1e-4).astype(F32)
    v0 = ((rng.standard_normal(n) * 1e-3) ** 2).astype(F32)
    hp = hparams(lr=0.0, weight_decay=0.01, step=3)
    m, v = m0.copy(), v0.copy()
    if fmt == "L12":
        G, W = oracle.bf16_from_f32(g32), oracle.bf16_from_f32(w32)
        W0 = W.copy()
        oracle.adamw_l12(G, W, m, v, hp)
        assert np.array_equal(W, W0)
    elif fmt == "L16M":
        G = oracle.bf16_from_f32(g32)
        master = w32.copy()
        Wb = np.zeros(n, np.uint16)
        oracle.adamw_l16m(G, master, m, v, Wb, hp)
        assert np.array_equal(master.view(np.uint32), w32.view(np.uint32))
        # the bf16 copy is the nearest-even rounding of the unchanged master
        import torch
        assert np.array_equal(Wb, torch.from_numpy(w32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    else:
        W = w32.copy()
        oracle.adamw_l16f(g32, W, m, v, hp)
        assert np.array_equal(W.view(np.uint32), w32.view(np.uint32))
    # the moments still advance
    assert not np.array_equal(m, m0) and not np.array_equal(v, v0)


@pytest.mark.parametrize("fmt", ["L16M", "L16F"])
def test_zero_gradient_is_pure_geometric_decay(fmt):
    """g = 0 and m = v = 0: the Adam step is exactly 0, so each step multiplies
    the fp32 weight by fl(1 - lr*wd) and nothing else."""
    n = 1000
    w0 = _weights(n, seed=9)
    lr, wd = 1e-2, 0.1
    d = F32(1.0 - lr * wd)
    W = w0.copy()
    m = np.zeros(n, F32)
    v = np.zeros(n, F32)
    Wb = np.zeros(n, np.uint16)
    expect = w0.copy()
    for t in range(1, 26):
        hp = hparams(lr=lr, weight_decay=wd, step=t)
        if fmt == "L16F":
            oracle.adamw_l16f(np.zeros(n, F32), W, m, v, hp)
        else:
            oracle.adamw_l16m(np.zeros(n, np.uint16), W, m, v, Wb, hp)
        expect = (expect * d).astype(F32)
        assert np.array_equal(W.view(np.uint32), expect.view(np.uint32)), t
        assert np.allclose(W, w0.astype(np.float64) * (1 - lr * wd) ** t, rtol=2 * t * U, atol=0)
    assert not np.any(m) and not np.any(v)


def test_zero_gradient_moments_decay_geometrically():
    """g = 0 with nonzero moments: m_t = b1^t m_0 and v_t = b2^t v_0, one fp32
    multiply per step (the (1-b)*g terms vanish)."""
    rng = np.random.default_rng(13)
    n = 777
    m0 = (rng.standard_normal(n) * 1e-4).astype(F32)
    v0 = ((rng.standard_normal(n) * 1e-3) ** 2).astype(F32)
    m, v = m0.copy(), v0.copy()
    W = _weights(n)
    em, ev = m0.copy(), v0.copy()
    for t in range(1, 11):
        oracle.adamw_l16f(np.zeros(n, F32), W, m, v, hparams(step=t))
        em = (em * F32(0.9)).astype(F32)
        ev = (ev * F32(0.999)).astype(F32)
        assert np.array_equal(m, em) and np.array_equal(v, ev), t


def test_decay_is_decoupled_and_applied_before_the_step():
    """AdamW reading: w' = w(1 - lr wd) - lr u. With lr = wd = 1/2, w = 1 and
    u = +-1 (t = 1, |g| >> eps) this is 0.75 -+ 0.5; decaying after the step
    would give 0.375 / 1.125, and an L2 term folded into g would give u = +-1
    with a different moment path."""
    g = np.array([0.5, -0.5], F32)
    W = np.array([1.0, 1.0], F32)
    m = np.zeros(2, F32)
    v = np.zeros(2, F32)
    oracle.adamw_l16f(g, W, m, v, hparams(lr=0.5, weight_decay=0.5, eps=1e-8, step=1))
    assert np.allclose(W, [0.25, 1.25], rtol=0, atol=1e-7)


# ---------------------------------------------------------------------------
# SGD: W_new = W_old - lr*g and W += (-lr*g) are the same operation
# ("The Assumption Everyone Makes").
# ---------------------------------------------------------------------------
def test_sgd_additive_form_equals_subtraction_fp32():
    rng = np.random.default_rng(17)
    n = 10007
    g = (rng.standard_normal(n)).astype(F32)
    w = (rng.standard_normal(n)).astype(F32)
    lr = F32(0.0173)
    W = w.copy()
    oracle.sgd_l16f(g, W, float(lr))
    traditional = (w - (lr * g).astype(F32)).astype(F32)
    assert np.array_equal(W.view(np.uint32), traditional.view(np.uint32))


def test_sgd_bf16_and_master_forms():
    import torch
    rng = np.random.default_rng(19)
    n = 5003
    g32 = (rng.standard_normal(n) * 1e-2).astype(F32)
    w32 = (rng.standard_normal(n) * 0.5).astype(F32)
    lr = 0.03
    Gb = torch.from_numpy(g32).to(torch.bfloat16)
    Wb = torch.from_numpy(w32).to(torch.bfloat16)
    # bf16 weights: widen, subtract in fp32, round to nearest even (torch's conversion)
    expect = (Wb.float() - (torch.tensor(lr, dtype=torch.float32) * Gb.float())).to(torch.bfloat16)
    W = Wb.view(torch.int16).numpy().view(np.uint16).copy()
    G = Gb.view(torch.int16).numpy().view(np.uint16).copy()
    oracle.sgd_l12(G, W, lr)
    assert np.array_equal(W, expect.view(torch.int16).numpy().view(np.uint16))
    # master form: fp32 master moves, bf16 copy is its rounding; no decay, no moments
    master = w32.copy()
    Wo = np.zeros(n, np.uint16)
    oracle.sgd_l16m(G, master, Wo, lr)
    em = (torch.from_numpy(w32) - torch.tensor(lr, dtype=torch.float32) * Gb.float())
    assert np.array_equal(master.view(np.uint32), em.numpy().view(np.uint32))
    assert np.array_equal(Wo, em.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


# ---------------------------------------------------------------------------
# bf16 rounding against an independent library conversion.
# ---------------------------------------------------------------------------
def test_bf16_round_nearest_even_matches_torch():
    import torch
    rng = np.random.default_rng(23)
    bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    hi = rng.integers(0, 2 ** 16, size=4096, dtype=np.uint64).astype(np.uint32) << 16
    specials = np.concatenate([
        hi | 0x8000, hi | 0x7FFF, hi | 0x8001, hi, hi | 0xFFFF,            # ties and neighbours
        np.array([0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0xFF7FFFFF,           # near the top: overflow to inf
                  0x00000001, 0x00008000, 0x00018000, 0x80008000,           # subnormals, ties
                  0x7F800000, 0xFF800000, 0x00000000, 0x80000000], np.uint32)])
    x = np.concatenate([bits, specials]).view(F32)
    mine = oracle.bf16_from_f32(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(mine[~nan], ref[~nan])
    back = oracle.f32_from_bf16(mine[nan])
    assert np.all(np.isnan(back))
    # widening is exact
    w = oracle.f32_from_bf16(ref[~nan])
    assert np.array_equal(w, torch.from_numpy(ref[~nan].view(np.int16)).view(torch.bfloat16).float().numpy())


def test_l12_and_l16m_are_the_fp32_update_on_widened_values():
    """The bf16 layouts apply the same per-element update to the widened bf16
    values; the bf16 outputs are the nearest-even roundings of the fp32 result."""
    rng = np.random.default_rng(29)
    n = 3001
    G = oracle.bf16_from_f32((rng.standard_normal(n) * 1e-3).astype(F32))
    Wb = oracle.bf16_from_f32((rng.standard_normal(n) * 0.02).astype(F32))
    m0 = (rng.standard_normal(n) * 1e-4).astype(F32)
    v0 = ((rng.standard_normal(n) * 1e-3) ** 2).astype(F32)
    hp = hparams(step=10)
    # fp32 layout on widened inputs
    Wf, mf, vf = oracle.f32_from_bf16(Wb), m0.copy(), v0.copy()
    oracle.adamw_l16f(oracle.f32_from_bf16(G), Wf, mf, vf, hp)
    # 12 B layout
    W12, m12, v12 = Wb.copy(), m0.copy(), v0.copy()
    oracle.adamw_l12(G, W12, m12, v12, hp)
    assert np.array_equal(m12, mf) and np.array_equal(v12, vf)
    assert np.array_equal(W12, oracle.bf16_from_f32(Wf))
    # 16 B mixed layout with master = widened W
    master, mm, vm, Wo = oracle.f32_from_bf16(Wb), m0.copy(), v0.copy(), np.zeros(n, np.uint16)
    oracle.adamw_l16m(G, master, mm, vm, Wo, hp)
    assert np.array_equal(master, Wf) and np.array_equal(Wo, oracle.bf16_from_f32(Wf))


# ---------------------------------------------------------------------------
# General t: the fp32 oracle is within a first-order rounding bound of the
# exact real-number result on the same fp32 inputs and fp32 step scalars.
# ---------------------------------------------------------------------------
getcontext().prec = 60


def _sqrt_frac(x: Fraction) -> Fraction:
    if x == 0:
        return Fraction(0)
    d = (Decimal(x.numerator) / Decimal(x.denominator)).sqrt()
    return Fraction(d)


def test_step_scalars_are_fp32_roundings_of_the_exact_values():
    for t in (1, 2, 10, 1000, 10 ** 6):
        for (b1, b2, lr, wd) in ((0.9, 0.999, 1e-4, 0.01), (0.95, 0.98, 3e-3, 0.1)):
            s = oracle.scalars(hparams(lr=lr, beta1=b1, beta2=b2, weight_decay=wd, step=t))
            # 60-digit decimal arithmetic on the fp32 hyperparameter values
            db1, db2 = Decimal(float(F32(b1))), Decimal(float(F32(b2)))
            dlr, dwd = Decimal(float(F32(lr))), Decimal(float(F32(wd)))
            for got, exact in ((s.bias_correction1, 1 - db1 ** t), (s.bias_correction2, 1 - db2 ** t),
                               (s.one_minus_beta1, 1 - db1), (s.one_minus_beta2, 1 - db2),
                               (s.decay, 1 - dlr * dwd)):
                e = float(exact)
                assert abs(got - e) <= float(np.spacing(F32(abs(e)))), (t, got, e)


@pytest.mark.parametrize("t", [1, 10, 1000])
def test_general_step_within_rounding_bound_of_exact(t):
    rng = np.random.default_rng(31 + t)
    n = 400
    g = (rng.standard_normal(n) * 1e-3).astype(F32)
    w = (rng.standard_normal(n) * 0.02).astype(F32)
    m0 = (rng.standard_normal(n) * 1e-4).astype(F32) if t > 1 else np.zeros(n, F32)
    v0 = ((rng.standard_normal(n) * 1e-3) ** 2).astype(F32) if t > 1 else np.zeros(n, F32)
    hp = hparams(lr=1e-4, weight_decay=0.01, step=t)
    s = oracle.scalars(hp)
    W, m, v = w.copy(), m0.copy(), v0.copy()
    oracle.adamw_l16f(g, W, m, v, hp)
    fr = lambda x: Fraction(float(x))
    b1, b2, o1, o2 = fr(s.beta1), fr(s.beta2), fr(s.one_minus_beta1), fr(s.one_minus_beta2)
    c1, c2, eps, lr, dec = (fr(s.bias_correction1), fr(s.bias_correction2), fr(s.eps), fr(s.lr),
                            fr(s.decay))
    for i in range(n):
        gi, wi, mi, vi = fr(g[i]), fr(w[i]), fr(m0[i]), fr(v0[i])
        mx = b1 * mi + o1 * gi
        vx = b2 * vi + o2 * gi * gi
        e_m = 2.01 * U * float(abs(b1 * mi) + abs(o1 * gi))
        e_v = 3.01 * U * float(abs(b2 * vi) + abs(o2 * gi * gi))
        assert abs(float(m[i]) - float(mx)) <= e_m + 1e-45
        assert abs(float(v[i]) - float(vx)) <= e_v + 1e-45
        mh, vh = mx / c1, vx / c2
        e_mh = e_m / float(c1) + U * abs(float(mh))
        e_vh = e_v / float(c2) + U * abs(float(vh))
        sq = _sqrt_frac(vh)
        e_sq = (e_vh / (2 * float(sq)) if sq > 0 else math.sqrt(e_vh)) + U * float(sq)
        den = sq + eps
        e_den = e_sq + U * float(den)
        u = mh / den
        e_u = e_mh / float(den) + abs(float(u)) * e_den / float(den) + U * abs(float(u))
        w1 = wi * dec
        st = lr * u
        wx = w1 - st
        e_w = U * abs(float(w1)) + float(lr) * e_u + U * abs(float(st)) + U * abs(float(wx))
        assert abs(float(W[i]) - float(wx)) <= 1.01 * e_w + 1e-45, (i, float(W[i]), float(wx), e_w)


# ---------------------------------------------------------------------------
# Gradient magnitude (progressive layer locking): sum of g^2 per block.
# ---------------------------------------------------------------------------
def test_grad_sq_closed_form_and_library():
    # g = k / 64 for k = 1..n: sum of squares = n(n+1)(2n+1)/6 / 4096, exact in fp64
    n = 2000
    g = (np.arange(1, n + 1) / 64.0).astype(F32)
    assert oracle.grad_sq(g) == n * (n + 1) * (2 * n + 1) / 6 / 4096
    gb = oracle.bf16_from_f32((np.arange(1, 201) / 8.0).astype(F32))  # exact in bf16
    assert oracle.grad_sq(gb) == 200 * 201 * 401 / 6 / 64
    rng = np.random.default_rng(41)
    x = (rng.standard_normal(100_000) * 1e-3).astype(F32)
    assert oracle.grad_sq(x) == pytest.approx(float(np.sum(x.astype(np.float64) ** 2)), rel=1e-12)
    xb = oracle.bf16_from_f32(x)
    assert oracle.grad_sq(xb) == pytest.approx(float(np.sum(oracle.f32_from_bf16(xb).astype(np.float64) ** 2)),
                                               rel=1e-12)
    assert oracle.grad_sq(np.zeros(0, F32)) == 0.0
