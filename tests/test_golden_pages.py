"""The pages' own worked examples and printed counts, against the oracle (CPU only)."""

import numpy as np
import pytest

import oracle
from oracle import hparams, layout
from synth import shapes

from conftest import load_golden

F32 = np.float32


def _floats(tokens):
    return np.array([float(x) for x in tokens], dtype=np.float64)


def _printed(values, d):
    """The values as the page prints them: fixed point with d decimals."""
    return [f"{float(x):.{d}f}" for x in values]


def test_m1_traditional_equals_frozen_sgd_reading():
    """Test 1: one reading that reproduces x 0.985 is SGD with g = W, lr = 0.015
    (loss W^2 / 2). Traditional: W - lr g. Frozen: W += (-lr g) (oracle)."""
    gold = load_golden("m1_equivalence.txt")
    d = int(gold["decimals"][0])
    w = _floats(gold["input"]).astype(F32)
    lr = 0.015
    traditional = (w - F32(lr) * w).astype(F32)
    frozen = w.copy()
    oracle.sgd_l16f(w.copy(), frozen, lr)
    assert _printed(traditional, d) == gold["traditional"]
    assert _printed(frozen, d) == gold["frozen"]
    assert np.array_equal(traditional.view(np.uint32), frozen.view(np.uint32))


def test_m1_adamw_reading_pure_decay():
    """The other reading: AdamW with zero gradient and zero moments and
    lr * wd = 0.015 is a pure x 0.985 decay. (Adam with g proportional to W and
    |g| >> eps would move every weight by about lr instead, which the printed
    values rule out: the example does not exercise the moment path.)"""
    gold = load_golden("m1_equivalence.txt")
    d = int(gold["decimals"][0])
    w = _floats(gold["input"]).astype(F32)
    W = w.copy()
    m = np.zeros(3, F32)
    v = np.zeros(3, F32)
    oracle.adamw_l16f(np.zeros(3, F32), W, m, v, hparams(lr=0.015, weight_decay=1.0, step=1))
    assert _printed(W, d) == gold["frozen"]
    # Adam with g = W: equal deltas, not proportional ones
    W2 = w.copy()
    oracle.adamw_l16f(w.copy(), W2, np.zeros(3, F32), np.zeros(3, F32),
                      hparams(lr=0.015, weight_decay=0.0, step=1))
    assert np.allclose(w - W2, 0.015, atol=1e-6)
    assert _printed(W2, d) != gold["frozen"]


def test_m2_additive_accumulation():
    """Test 2: [1, 2] += [0.5, 0.3] gives [1.5, 2.3]; the additive apply is
    SGD's W += (-lr g) with lr = 1 and g = -delta."""
    gold = load_golden("m2_accumulation.txt")
    d = int(gold["decimals"][0])
    W = _floats(gold["first"]).astype(F32)
    delta = _floats(gold["delta"]).astype(F32)
    oracle.sgd_l16f(-delta, W, 1.0)
    assert _printed(W, d) == gold["result"]


# ---------------------------------------------------------------------------
# Printed counts and byte totals against the oracle's block calculator.
# ---------------------------------------------------------------------------
def _g(key):
    return load_golden("param_counts.txt")[key][0]


def test_llama7b_counts_and_bytes():
    L = layout.plan(shapes.llama7b(), "L16M")
    n = L.n_params
    assert n == int(_g("llama7b_params"))
    assert round(n * 16 / 1e9, 1) == float(_g("llama7b_total_gb_16B"))
    assert round(n * 2 / 1e9, 1) == float(_g("llama7b_weights_gb_2B"))
    assert round(n * 4 / 1e9, 1) == float(_g("llama7b_master_gb_4B"))
    assert round(n * 8 / 1e9, 1) == float(_g("llama7b_optimizer_gb_8B"))
    assert len(L.blocks) == 34
    # every block holds 16 B per padded element in the mixed layout
    assert all(b.nbytes == 16 * b.padded for b in L.blocks)


def test_toy_decoder_state_bytes():
    n = int(_g("toy_decoder_params"))
    assert n * 16 == int(_g("toy_decoder_state_bytes"))


def test_tinyllama_base_and_lora_counts():
    base = layout.plan(shapes.tinyllama_full(), "L16M")
    assert round(base.n_params / 1e9, 2) == float(_g("tinyllama_base_params_billions"))
    assert round(base.n_params * 2 / 1e9, 2) == float(_g("tinyllama_base_gb_bf16"))
    lo = layout.plan(shapes.tinyllama_lora(8), "L16F")
    assert round(lo.n_params / 1e6, 1) == float(_g("tinyllama_lora_params_millions"))
    assert round(100 * lo.n_params / base.n_params, 2) == float(_g("tinyllama_lora_percent"))
    assert round(lo.n_params * 4 / 1e6, 2) == float(_g("tinyllama_lora_adapters_mb"))
    assert round(lo.n_params * 8 / 1e6, 2) == float(_g("tinyllama_lora_adam_mb"))
    assert sum(len(b.spans) for b in lo.blocks) == 7 * 2 * 22


def test_seventy_b_byte_arithmetic():
    """Page 1's 782 GB are GiB of W, M, V in fp32 (12 B/param); its 3.5 GB per
    layer is 70B/80 fp32 weights; page 4's 840 GB are decimal GB at 12 B/param;
    120B at 12 B/param is about 1.5 TB."""
    assert round(70e9 * 12 / 2 ** 30) == int(_g("seventy_b_files_gib_12B"))
    assert round(70e9 / 80 * 4 / 1e9, 1) == float(_g("seventy_b_layer_gb_4B"))
    assert round(70e9 * 12 / 1e9) == int(_g("seventy_b_state_gb_12B"))
    # 1.44 TB, printed as "about 1.5 TB"
    assert 120e9 * 12 / 1e12 == pytest.approx(float(_g("onetwenty_b_state_tb_12B")), abs=0.07)
    # a Llama-70B decoder layer is within 3% of the page's 70B / 80 per layer
    L = layout.plan(shapes.llama70b_slice(1), "L12")
    assert abs(L.n_params - 70e9 / 80) / (70e9 / 80) < 0.03


def test_layout_geometry_rules():
    for fmt, bpp in (("L12", 12), ("L16M", 16), ("L16F", 16)):
        for specs in (shapes.tinyllama_layer(), shapes.tinyllama_lora(), [("a", (1,), 0), ("b", (7,), 0),
                                                                          ("c", (9,), 1), ("d", (4097,), 1)]):
            L = layout.plan(specs, fmt)
            for b in L.blocks:
                assert b.padded % 2048 == 0 and b.nbytes == bpp * b.padded
                for (off, size) in b.segments.values():
                    assert off % 4096 == 0 and size % 4096 == 0
                for (_, off, n) in b.spans:
                    assert off % 8 == 0
                # spans do not overlap and stay inside the block
                ends = sorted((off, off + n) for (_, off, n) in b.spans)
                for (a0, a1), (b0, b1) in zip(ends, ends[1:]):
                    assert a1 <= b0
                assert ends[-1][1] <= b.padded
                # the input prefix and output suffix are contiguous ranges
                assert b.h2d[0] == 0
                assert b.d2h[0] + b.d2h[1] == b.nbytes


def test_tiny_odd_shapes_padding():
    L = layout.plan([("a", (1,), 0), ("b", (7,), 0), ("c", (9,), 0), ("d", (4097,), 0)], "L12")
    b = L.blocks[0]
    assert [off for (_, off, _) in b.spans] == [0, 8, 16, 32]
    assert b.params == 1 + 7 + 9 + 4097
    assert b.padded == 6144
