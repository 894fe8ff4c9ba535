"""The C ABI without a GPU: exported symbols, block geometry (bit-exact against
the oracle's calculator), argument validation that happens before any CUDA
call, status strings."""

import ctypes
import json
import os
import re

import pytest

from conftest import ROOT
from oracle import layout as olayout
from synth import shapes


@pytest.fixture(scope="module")
def L():
    from optimizer_update_gb300 import lst
    if not os.path.exists(lst.LIB_PATH):
        from optimizer_update_gb300 import build
        build.build()
    return lst


def _declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "lst.h")).read()
    return sorted(set(re.findall(r"^LST_API [^;]*?\b(lst_\w+)\(", hdr, flags=re.M)))


def test_library_exports_every_declared_symbol(L):
    names = _declared_symbols()
    assert len(names) >= 16
    raw = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def _edge_specs():
    return [
        ("scalar", (), 0), ("one", (1,), 0), ("seven", (7,), 0), ("nine", (3, 3), 0),
        ("tail", (4097,), 1), ("empty", (0, 5), 1), ("four_d", (2, 3, 4, 5), 1),
    ]


CASES = [(n, fn, fmt) for n, (fn, fmt) in shapes.WORKLOADS.items()] + [
    ("edge_l12", _edge_specs, "L12"), ("edge_l16m", _edge_specs, "L16M"), ("edge_l16f", _edge_specs, "L16F"),
    ("lora_as_l12", shapes.tinyllama_lora, "L12"), ("layer_as_l16m", shapes.tinyllama_layer, "L16M"),
]


@pytest.mark.parametrize("name,fn,fmt", CASES, ids=[c[0] for c in CASES])
def test_layout_geometry_matches_oracle_bit_exact(L, name, fn, fmt):
    specs = fn()
    O = olayout.plan(specs, fmt)
    h = L.lst_layout_create([s for (_, s, _) in specs], [l for (_, _, l) in specs], fmt)
    try:
        n_layers, n_params, max_bytes = L.lst_layout_info(h)
        assert (n_layers, n_params, max_bytes) == (len(O.blocks), O.n_params, O.max_block_bytes)
        for i, b in enumerate(O.blocks):
            assert L.lst_layout_block(h, i) == (b.nbytes, b.params, b.padded)
            for f, (off, size) in b.segments.items():
                assert L.lst_layout_segment(h, i, f) == (off, size)
            assert L.lst_layout_transfer(h, i) == (b.h2d[0], b.h2d[1], b.d2h[0], b.d2h[1])
        for t in range(len(specs)):
            for f in O.blocks[O.tensor_block[t]].segments:
                off, layer, eoff = L.lst_layout_tensor(h, t, f)
                assert off == O.tensor_byte_offset(t, f)
                assert (layer, eoff) == (O.tensor_block[t], O.tensor_elem_offset[t])
    finally:
        L.lst_layout_destroy(h)


def test_empty_layout(L):
    h = L.lst_layout_create([], [], "L12")
    assert L.lst_layout_info(h) == (0, 0, 0)
    # a step over no blocks is a no-op and needs no device
    L.lst_adamw_step(h, [], L.adamw_hparams(step=1))
    L.lst_layout_destroy(h)


@pytest.mark.parametrize("shapes_,layers,fmt", [
    ([(1, 2, 3, 4, 5)], [0], "L12"),     # ndim 5
    ([(-1,)], [0], "L12"),               # negative dim
    ([(4,), (4,)], [0, 2], "L12"),       # block 1 has no tensors
    ([(4,)], [-1], "L12"),               # negative block
    ([(4,)], [0], 7),                    # unknown format
    ([(1 << 21, 1 << 20)], [0], "L12"),  # 2^41 elements
])
def test_layout_create_rejects(L, shapes_, layers, fmt):
    with pytest.raises(L.LstError) as e:
        L.lst_layout_create(shapes_, layers, fmt)
    assert e.value.status == L.LST_ERR_INVALID_ARG


def test_geometry_queries_reject_out_of_range(L):
    h = L.lst_layout_create([(8,)], [0], "L12")
    try:
        for call in (lambda: L.lst_layout_block(h, 1), lambda: L.lst_layout_segment(h, 0, "MASTER"),
                     lambda: L.lst_layout_tensor(h, 1, "G"), lambda: L.lst_layout_transfer(h, -1),
                     lambda: L.lst_layout_set_stream_chunk(h, 1000),
                     lambda: L.lst_layout_set_stream_copy(h, 3, 0), lambda: L.lst_layout_set_stream_copy(h, 0, -1),
                     lambda: L.lst_stream_copy_choice(h, 1), lambda: L.lst_stream_copy_choice(h, -1)):
            with pytest.raises(L.LstError) as e:
                call()
            assert e.value.status == L.LST_ERR_INVALID_ARG
        L.lst_layout_set_stream_chunk(h, 4096)
        L.lst_layout_set_stream_chunk(h, 0)
        # no streamed step has run: no statistics yet
        assert L.lst_stream_last_stats(h) == {f: 0 for f, _ in L.lst_stream_stats._fields_}
        # no streamed step has timed the block yet: nothing learned
        c = L.lst_stream_copy_choice(h, 0)
        assert not c["measured"] and c["chunks"] == 0 and c["kernel_in_chunks"] == 0
        for a in (L.LST_COPY_ENGINE, L.LST_COPY_SM, L.LST_COPY_AUTO):
            for b in (L.LST_COPY_ENGINE, L.LST_COPY_SM, L.LST_COPY_AUTO):
                L.lst_layout_set_stream_copy(h, a, b)
                assert not L.lst_stream_copy_choice(h, 0)["measured"]
    finally:
        L.lst_layout_destroy(h)


def test_step_validation_before_any_cuda_call(L):
    h = L.lst_layout_create([(8,)], [0], "L12")
    try:
        bad = [L.adamw_hparams(step=0), L.adamw_hparams(beta1=1.0), L.adamw_hparams(beta2=-0.1),
               L.adamw_hparams(lr=float("nan")), L.adamw_hparams(eps=float("inf"))]
        for hp in bad:
            with pytest.raises(L.LstError) as e:
                L.lst_adamw_step(h, [4096], hp)
            assert e.value.status == L.LST_ERR_INVALID_ARG
            with pytest.raises(L.LstError) as e:
                L.lst_stream_step(h, [4096], 4096, 8192, hp)
            assert e.value.status == L.LST_ERR_INVALID_ARG
        with pytest.raises(L.LstError) as e:
            L.lst_adamw_step(h, [4096 + 8], L.adamw_hparams())
        assert e.value.status == L.LST_ERR_ALIGNMENT
        with pytest.raises(L.LstError) as e:
            L.lst_adamw_step(h, [0], L.adamw_hparams())
        assert e.value.status == L.LST_ERR_INVALID_ARG
        with pytest.raises(L.LstError) as e:
            L.lst_sgd_step(h, [4096], float("inf"))
        assert e.value.status == L.LST_ERR_INVALID_ARG
        with pytest.raises(L.LstError) as e:
            L.lst_stream_step(h, [4096 + 64], 4096, 8192, L.adamw_hparams())
        assert e.value.status == L.LST_ERR_ALIGNMENT
        with pytest.raises(L.LstError) as e:
            L.lst_stream_step(h, [4096], 4096 + 16, 8192, L.adamw_hparams())
        assert e.value.status == L.LST_ERR_ALIGNMENT
        with pytest.raises(L.LstError) as e:
            L.lst_stream_step(h, [4096], 0, 8192, L.adamw_hparams())
        assert e.value.status == L.LST_ERR_INVALID_ARG
    finally:
        L.lst_layout_destroy(h)


def test_status_strings_and_inject_validation(L):
    for st in range(7):
        assert L.lst_status_string(st)
    assert L.lst_status_string(99) == "unknown status"
    with pytest.raises(L.LstError):
        L.lst_test_inject(5, 0)
    with pytest.raises(L.LstError):
        L.lst_test_inject(1, 0)
    L.lst_test_inject(0, 0)
    assert L.lst_last_error() == ""


def test_product_does_not_reach_the_oracle():
    """The product package never imports, loads or names the oracle."""
    pkg = os.path.join(ROOT, "optimizer_update_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f
                assert "synth" not in text, f


def test_step_options_validation_before_any_cuda_call(L):
    h = L.lst_layout_create([(8,), (8,)], [0, 1], "L12")
    try:
        assert L.lst_workspace_bytes() == 256 + 8 * 1024 * 128
        with pytest.raises(L.LstError) as e:  # a block step of 0
            L.lst_adamw_step_ex(h, [4096, 8192], L.adamw_hparams(), L.step_options(block_steps=[1, 0]))
        assert e.value.status == L.LST_ERR_INVALID_ARG
        with pytest.raises(L.LstError) as e:  # grad_sq without a workspace
            L.lst_adamw_step_ex(h, [4096, 8192], L.adamw_hparams(), L.step_options(grad_sq=4096))
        assert e.value.status == L.LST_ERR_INVALID_ARG
        with pytest.raises(L.LstError) as e:  # misaligned workspace
            L.lst_adamw_step_ex(h, [4096, 8192], L.adamw_hparams(), L.step_options(grad_sq=4096, workspace=4096 + 64))
        assert e.value.status == L.LST_ERR_ALIGNMENT
        # a skipped block's bad step counter is never looked at; all blocks skipped: nothing to do
        L.lst_adamw_step_ex(h, [0, 0], L.adamw_hparams(), L.step_options(block_steps=[0, 0], skip=[1, 1]))
        with pytest.raises(L.LstError) as e:
            L.lst_stream_step_ex(h, [4096, 8192], 4096, 8192, L.adamw_hparams(), L.step_options(block_steps=[0, 1]))
        assert e.value.status == L.LST_ERR_INVALID_ARG
    finally:
        L.lst_layout_destroy(h)


def test_gradient_event_step_validation_before_any_cuda_call(L):
    """lst_stream_step_devgrad_events refuses an order that is not a
    permutation of the blocks, and missing gradients, before any CUDA call
    (the pointers below are never dereferenced)."""
    h = L.lst_layout_create([(8,), (8,), (8,)], [0, 1, 2], "L12")
    try:
        hosts, grads, evs = [4096, 8192, 12288], [256, 512, 768], [0, 0, 0]
        for order in ([0, 0, 1], [0, 1, 3], [2, 1, -1]):
            with pytest.raises(L.LstError) as e:
                L.lst_stream_step_devgrad_events(h, hosts, grads, evs, order, 4096, 8192, L.adamw_hparams())
            assert e.value.status == L.LST_ERR_INVALID_ARG and "permutation" in str(e.value)
        with pytest.raises(L.LstError) as e:  # a gradient pointer missing
            L.lst_stream_step_devgrad_events(h, hosts, [256, 0, 768], evs, [2, 1, 0], 4096, 8192,
                                             L.adamw_hparams())
        assert e.value.status == L.LST_ERR_INVALID_ARG
        with pytest.raises(L.LstError) as e:  # a misaligned gradient
            L.lst_stream_step_devgrad_events(h, hosts, [256, 520, 768], evs, None, 4096, 8192, L.adamw_hparams())
        assert e.value.status == L.LST_ERR_ALIGNMENT
        r = L.lib().lst_stream_step_devgrad_events(h, L._ptr_array(hosts), None, L._ptr_array(evs), None,
                                                   4096, 8192, ctypes.byref(L.adamw_hparams()), None, 0)
        assert r == L.LST_ERR_INVALID_ARG  # no gradients at all
    finally:
        L.lst_layout_destroy(h)


def test_bench_runs_the_oracle_only_in_its_baseline_and_reference_legs():
    """bench.py imports the oracle only inside the CPU-baseline helpers and the
    reference arm, and calls those helpers only from the baseline leg (rank 0,
    one process, CPU baseline on) and from the reference entry."""
    import ast
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    importers = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in node.names):
                    importers.add(fn.name)
                if isinstance(node, ast.ImportFrom) and (node.module or "").split(".")[0] == "oracle":
                    importers.add(fn.name)
    assert importers == {"cpu_oracle_rate", "parity_sample", "parity_stream", "run_reference"}
    # no module-level import of the oracle
    for node in tree.body:
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            names = [a.name for a in node.names] + [getattr(node, "module", None) or ""]
            assert not any(n.split(".")[0] == "oracle" for n in names)
    # the baseline helpers are called only under the CPU-baseline condition
    src = open(os.path.join(ROOT, "bench.py")).read()
    for helper in ("cpu_oracle_rate(", "parity_sample(", "parity_stream("):
        calls = [i for i in range(len(src)) if src.startswith(helper, i) and not src[:i].endswith("def ")]
        assert len(calls) == 1, helper
        guard = src.rfind("if rank == 0 and world == 1 and not args.no_cpu_baseline:", 0, calls[0])
        assert guard != -1 and calls[0] - guard < 800, helper


def test_bench_reference_arm_uses_only_the_oracle_and_the_generator():
    """bench.py --impl reference builds its geometry, inputs and steps from
    oracle/ and synth/ alone: the product library is never imported or
    loaded in that process (a 4 MiB sample of the Llama-70B slice's first
    block, one timed step)."""
    import subprocess
    import sys
    code = (
        "import sys, json\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "rc = bench.main(['--impl', 'reference', '--steps', '1', '--warmup', '3', '--ref-step-s', '0.01',"
        " '--ref-sample-bytes', str(4 << 20)])\n"
        "maps = open('/proc/self/maps').read()\n"
        "print('LOADED', 'liblst.so' in maps, 'optimizer_update_gb300' in sys.modules)\n"
        "sys.exit(rc)\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.strip().splitlines()
    line = json.loads([x for x in lines if x.startswith("{")][0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["name"] == "llama70b_slice8_l12"
    assert "first" in line["cpu_baseline"]["sample"]
    assert lines[-1] == "LOADED False False"


def test_bench_health_check_flags_either_direction():
    """The bench's pinned-state health check: a block counts as slow when
    either direction is under 0.85 of the best block's rate in that direction."""
    import bench
    h2d = [210.0, 200.0, 20.0, 209.0]
    d2h = [193.0, 150.0, 193.0, 192.0]
    assert bench.slow_block_flags((h2d, d2h)) == [False, True, True, False]
    assert bench.slow_block_flags((h2d, d2h), frac=0.7) == [False, False, True, False]


def test_bench_copy_choice_summary_adds_up_blocks():
    """The bench's summary of what the default copy mode learned: sums over
    the measured blocks, minima over the rates that were timed."""
    import bench

    class FakeLayout:
        n_layers = 3
        _c = [dict(measured=True, chunks=10, kernel_in_chunks=2, kernel_out_chunks=0, engine_h2d_gbs_min=4.5,
                   engine_h2d_gbs_max=200.0, engine_d2h_gbs_min=150.0, engine_d2h_gbs_max=190.0),
              dict(measured=False, chunks=0, kernel_in_chunks=0, kernel_out_chunks=0, engine_h2d_gbs_min=0.0,
                   engine_h2d_gbs_max=0.0, engine_d2h_gbs_min=0.0, engine_d2h_gbs_max=0.0),
              dict(measured=True, chunks=4, kernel_in_chunks=4, kernel_out_chunks=1, engine_h2d_gbs_min=0.0,
                   engine_h2d_gbs_max=0.0, engine_d2h_gbs_min=120.0, engine_d2h_gbs_max=180.0)]

        def stream_copy_choice(self, i):
            return self._c[i]

    s = bench.copy_choice_summary(FakeLayout())
    assert s == {"blocks_measured": 2, "chunks": 14, "kernel_in_chunks": 6, "kernel_out_chunks": 1,
                 "engine_h2d_gbs_min": 4.5, "engine_d2h_gbs_min": 120.0}
