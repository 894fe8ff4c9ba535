"""The seeded input generator: determinism, random access, scales (CPU only)."""

import numpy as np

import synth
from oracle import layout
from synth import shapes


def test_counter_based_random_access_matches_fill():
    a = np.empty(5000, np.float32)
    synth.fill(a, synth.KIND_F32, 7, synth.stream_id(synth.FIELD_G, 3), 1000, 1e-3)
    idx = np.array([1000, 1001, 3333, 5999], np.uint64)
    b = synth.gather(synth.KIND_F32, 7, synth.stream_id(synth.FIELD_G, 3), idx, 1e-3)
    assert np.array_equal(b, a[idx.astype(np.int64) - 1000])


def test_threads_do_not_change_values():
    a = np.empty(3_000_001, np.uint16)
    b = np.empty(3_000_001, np.uint16)
    synth.fill(a, synth.KIND_BF16, 1, 2, 0, 0.02, threads=1)
    synth.fill(b, synth.KIND_BF16, 1, 2, 0, 0.02, threads=7)
    assert np.array_equal(a, b)


def test_scale_and_moments():
    a = np.empty(1 << 22, np.float32)
    synth.fill(a, synth.KIND_F32, 11, 5, 0, 0.02)
    assert abs(a.std() - 0.02) < 2e-4 and abs(a.mean()) < 1e-4
    assert np.abs(a).max() <= 0.02 * 3.47
    q = np.empty(1 << 20, np.float32)
    synth.fill(q, synth.KIND_SQ_F32, 11, 6, 0, 1e-3)
    assert np.all(q >= 0) and abs(q.mean() - 1e-6) < 2e-8


def test_bf16_is_upper_half_of_f32():
    f = np.empty(4096, np.float32)
    h = np.empty(4096, np.uint16)
    synth.fill(f, synth.KIND_F32, 3, 9, 17, 0.5)
    synth.fill(h, synth.KIND_BF16, 3, 9, 17, 0.5)
    assert np.array_equal(h, (f.view(np.uint32) >> 16).astype(np.uint16))


def test_different_streams_and_seeds_differ():
    a = np.empty(1024, np.float32)
    b = np.empty(1024, np.float32)
    synth.fill(a, synth.KIND_F32, 1, synth.stream_id(1, 0), 0, 1.0)
    synth.fill(b, synth.KIND_F32, 1, synth.stream_id(1, 1), 0, 1.0)
    assert not np.array_equal(a, b)
    synth.fill(b, synth.KIND_F32, 2, synth.stream_id(1, 0), 0, 1.0)
    assert not np.array_equal(a, b)


def test_fill_block_and_gather_block_agree_with_zero_padding():
    specs = [("a", (3, 5), 0), ("b", (7,), 0), ("lora_B", (9, 2), 0)]
    for fmt in ("L12", "L16M", "L16F"):
        L = layout.plan(specs, fmt)
        blk = L.blocks[0]
        fields = {f: np.full(blk.padded, 77, np.uint16 if dt == "bf16" else np.float32)
                  for f, dt in synth.FORMAT_FIELDS[fmt]}
        synth.fill_block(fields, blk.spans, 0, "tinyllama_lora_l16f", fmt, t=10)
        used = np.zeros(blk.padded, bool)
        for (_, off, n) in blk.spans:
            used[off:off + n] = True
        idx = np.arange(blk.padded)
        for f, dt in synth.FORMAT_FIELDS[fmt]:
            assert not np.any(fields[f][~used])  # padding is zero
            g = synth.gather_block(f, fmt, blk.spans, 0, "tinyllama_lora_l16f", 10, idx)
            assert np.array_equal(g, fields[f])


def test_recipe_zero_moments_at_step_one():
    specs = shapes.tinyllama_lora()[:4]
    L = layout.plan(specs, "L16F")
    blk = L.blocks[0]
    fields = {f: np.ones(blk.padded, np.float32) for f, _ in synth.FORMAT_FIELDS["L16F"]}
    synth.fill_block(fields, blk.spans, 0, "tinyllama_lora_l16f", "L16F", t=1)
    assert not np.any(fields["M"]) and not np.any(fields["V"])
    for (name, off, n) in blk.spans:
        if name.endswith("lora_B"):
            assert not np.any(fields["W"][off:off + n])
        else:
            assert np.any(fields["W"][off:off + n])
