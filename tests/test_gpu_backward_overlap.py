"""The streamed step overlapped with a backward pass that produces the gradients (GB300).

The "MegaTrain" summary page (three-stream execution) releases each layer's
gradient with a Backward-Done event. Here a gradient producer on the device
(the input generator's GPU twin, synth/gen_dev.cu, standing in for backward)
writes block i's gradient on its own stream and records an event; the
streamed step (lst_stream_step_devgrad_events) streams each block's state in
without waiting, and lets block i's update wait on the device for its event.
The blocks go last to first, as backward finishes them.

The gradient buffers start as NaN and the producer is made slow (extra hash
rounds per element), so an update that did not wait would read NaN: results
are compared with the oracle, bit for bit, on the generator's gradient.
"""

import numpy as np
import pytest

import oracle
import synth
from optimizer_update_gb300 import Layout, lst
from synth import shapes

from gpu_util import SEED, PinnedBlocks, compare, fill_host_block, hparams_for, oracle_step

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SLOW = 200  # hash rounds per element: the producer takes several times a block's copy-in time


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    lst.lst_test_inject(0, 0)
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", [synth.KIND_BF16, synth.KIND_F32, synth.KIND_SQ_F32])
@pytest.mark.parametrize("passes", [1, 7])
def test_device_generator_matches_the_host_generator(kind, passes):
    n, start, stream_id, sigma = (1 << 20) + 37, 123_457, synth.stream_id(synth.FIELD_G, 5), 1e-3
    host = np.empty(n, np.uint16 if kind == synth.KIND_BF16 else np.float32)
    synth.fill(host, kind, SEED, stream_id, start, sigma)
    dev = torch.empty(host.nbytes, dtype=torch.uint8, device="cuda")
    rc = synth.dev_lib().synth_dev_fill(kind, SEED, stream_id, start, n, float(synth.scale_for(sigma)),
                                        dev.data_ptr(), passes, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(dev.cpu().numpy(), host.view(np.uint8))


@pytest.mark.parametrize("fmt,workload", [("L12", "tinyllama_layer_l12"), ("L16F", "tinyllama_lora_l16f")])
def test_device_gradient_field_matches_fill_field(fmt, workload):
    specs = [(n, sh, 0) for (n, sh, _) in shapes.tinyllama_layer()] + [("odd", (4097,), 0)]
    L = Layout(specs, fmt)
    host = np.full(L.block_bytes(0), 0x55, np.uint8)
    views = L.numpy_views(0, host)
    synth.fill_field(views["G"], "G", fmt, L.spans(0), 0, workload, 10)
    off, nbytes = L.segment(0, "G")
    dev = torch.full((nbytes,), 0x55, dtype=torch.uint8, device="cuda")
    synth.device_fill_field(dev.data_ptr(), "G", fmt, L.spans(0), L.padded(0), 0, workload, 10, SEED,
                            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(dev.cpu().numpy(), host[off:off + nbytes])


def _layers():
    specs = [(n, sh, l - 1) for (n, sh, l) in shapes.tinyllama_full() if l in (1, 2, 3)]
    return specs + [("odd", (4097,), 1), ("odder", (9,), 2), ("last", (70_001,), 3)]


def _produce(L, grads, events, order, workload, t, g_seed, stream, passes):
    """The backward stand-in: block by block in `order`, write the gradient
    and record the block's Backward-Done event on the producer stream."""
    with torch.cuda.stream(stream):
        for i in order:
            synth.device_fill_field(grads[i].data_ptr(), "G", L.fmt, L.spans(i), L.padded(i), i, workload, t,
                                    g_seed, stream.cuda_stream, passes)
            events[i].record(stream)


@pytest.mark.parametrize("fmt,workload", [("L12", "tinyllama_layer_l12"), ("L16M", "tinyllama_full_l16m"),
                                          ("L16F", "tinyllama_lora_l16f")])
@pytest.mark.parametrize("chunk", [0, 1 << 20])
def test_overlapped_step_matches_the_oracle(fmt, workload, chunk):
    L = Layout(_layers(), fmt)
    L.set_stream_chunk(chunk)
    n = L.n_layers
    order = list(reversed(range(n)))
    P = PinnedBlocks(L, guard=4096)
    try:
        for i in range(n):
            fill_host_block(L, i, P.arrays[i], workload, 10)
        ref = [a.copy() for a in P.arrays]
        poison = []
        for i in range(n):  # the host gradient segments are neither read nor written
            g = L.numpy_views(i, P.arrays[i])["G"].view(np.uint8)
            g[:] = 0x7F
            poison.append(g.copy())
        grads = [torch.full((L.segment(i, "G")[1],), 0xFF, dtype=torch.uint8, device="cuda") for i in range(n)]
        b0 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        b1 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        producer = torch.cuda.Stream()
        for k, t in enumerate((10, 11)):
            g_seed = SEED + 1000 * k
            events = [torch.cuda.Event() for _ in range(n)]
            if k:  # the next step's gradient, into NaN-filled buffers again
                for g in grads:
                    g.fill_(0xFF)
            producer.wait_stream(torch.cuda.current_stream())
            _produce(L, grads, events, order, workload, t, g_seed, producer, SLOW)
            hp, ohp = hparams_for(workload, t)
            lst.lst_stream_step_devgrad_events(L.handle, P.ptrs, [g.data_ptr() for g in grads],
                                               [e.cuda_event for e in events], order, b0.data_ptr(), b1.data_ptr(),
                                               hp, None, 600_000)
            for i in range(n):
                synth.fill_field(L.numpy_views(i, ref[i])["G"], "G", fmt, L.spans(i), i, workload, t, g_seed)
                oracle_step(L, ref[i], i, ohp)
        torch.cuda.synchronize()
        assert P.guards_intact(), "write outside a host block"
        for i in range(n):
            got, exp = L.numpy_views(i, P.arrays[i]), L.numpy_views(i, ref[i])
            assert np.array_equal(got["G"].view(np.uint8), poison[i])
            for f in got:
                if f != "G":
                    assert np.array_equal(got[f].view(np.uint8), exp[f].view(np.uint8)), (i, f)
            compare(fmt, got, exp)
    finally:
        P.free()


def test_overlapped_step_with_options_and_ready_gradients():
    """Per-block step counters, a locked block, sums of g^2, and a mix of
    events and NULL entries (gradients already complete), in a shuffled
    order."""
    fmt, workload = "L16M", "tinyllama_full_l16m"
    L = Layout(_layers(), fmt)
    L.set_stream_chunk(1 << 21)
    n = L.n_layers
    order = [2, 0, 3, 1][:n]
    skip = [0, 1, 0, 0][:n]
    steps = [12, 5, 9, 30][:n]
    P = PinnedBlocks(L)
    try:
        for i in range(n):
            fill_host_block(L, i, P.arrays[i], workload, 10)
        ref = [a.copy() for a in P.arrays]
        grads = [torch.full((L.segment(i, "G")[1],), 0xFF, dtype=torch.uint8, device="cuda") for i in range(n)]
        producer = torch.cuda.Stream()
        producer.wait_stream(torch.cuda.current_stream())
        # odd blocks: gradient complete before the call (a NULL entry)
        with torch.cuda.stream(producer):
            for i in range(1, n, 2):
                synth.device_fill_field(grads[i].data_ptr(), "G", fmt, L.spans(i), L.padded(i), i, workload, 10,
                                        SEED, producer.cuda_stream)
        producer.synchronize()
        # even blocks: produced slowly while the step runs, each behind its event
        events = [torch.cuda.Event() for _ in range(n)]
        _produce(L, grads, events, [i for i in order if i % 2 == 0], workload, 10, SEED, producer, SLOW)
        ready = [events[i].cuda_event if i % 2 == 0 else 0 for i in range(n)]
        gsq = torch.full((n,), -1.0, dtype=torch.float64, device="cuda")
        ws = torch.empty(lst.lst_workspace_bytes(), dtype=torch.uint8, device="cuda")
        b0 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        b1 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        hp, _ = hparams_for(workload, 10)
        opts = lst.step_options(block_steps=steps, skip=skip, grad_sq=gsq.data_ptr(), workspace=ws.data_ptr())
        lst.lst_stream_step_devgrad_events(L.handle, P.ptrs, [g.data_ptr() for g in grads], ready, order,
                                           b0.data_ptr(), b1.data_ptr(), hp, opts, 600_000)
        g = gsq.cpu().numpy()
        for i in range(n):
            if skip[i]:
                assert np.array_equal(P.arrays[i], ref[i]) and g[i] == -1.0
                continue
            exp_sq = oracle.grad_sq(L.numpy_views(i, ref[i])["G"])
            assert abs(g[i] - exp_sq) <= 1e-6 * exp_sq, (i, g[i], exp_sq)
            oracle_step(L, ref[i], i, hparams_for(workload, steps[i])[1])
            got, exp = L.numpy_views(i, P.arrays[i]), L.numpy_views(i, ref[i])
            for f in got:
                if f != "G":
                    assert np.array_equal(got[f].view(np.uint8), exp[f].view(np.uint8)), (i, f)
    finally:
        P.free()
