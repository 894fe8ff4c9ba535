"""The step variant for callers that cannot allocate device memory (GB300).

Some callers have no way to allocate device memory when they step the
optimizer (their device memory belongs to another allocator, or they must not
allocate once running), so they cannot pass the workspace the per-block
sum-of-squares reduction needs. lst_adamw_step_ex_noalloc uses a static
device array of the library instead. This file checks, through the C ABI,
that it gives the same results as lst_adamw_step_ex with a caller workspace,
on two calls in a row (the second call finds the array holding the first
call's partial sums), including a step over more blocks than one launch's
partial sums fill, and that a call refused by validation touches nothing.
It is named to be collected last, and passes on its own in a fresh process
as well as after the other tests.
"""

import numpy as np
import pytest

import oracle
from optimizer_update_gb300 import Layout, lst
from synth import shapes

from gpu_util import compare, fill_host_block, hparams_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GSQ_REL = 1e-6  # as the per-block options tests: 7 fp32 roundings of a nonnegative sum < 5e-7


@pytest.fixture(autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    yield
    torch.cuda.synchronize()


def _specs():
    s = [(n, sh, l - 1) for (n, sh, l) in shapes.tinyllama_full() if l in (1, 2)]
    return s + [("odd", (4097,), 2), ("tiny", (9,), 3), ("lora_A", (8, 2048), 4), ("lora_B", (2048, 8), 4)]


@pytest.mark.parametrize("fmt,workload", [("L16M", "tinyllama_full_l16m"), ("L12", "tinyllama_layer_l12")])
def test_noalloc_matches_the_workspace_variant_on_two_calls(fmt, workload):
    L = Layout(_specs(), fmt)
    hosts = [np.empty(L.block_bytes(i), np.uint8) for i in range(L.n_layers)]
    for i in range(L.n_layers):
        fill_host_block(L, i, hosts[i], workload, 10)
    a = [torch.from_numpy(h).cuda() for h in hosts]   # stepped by the no-allocation variant
    b = [torch.from_numpy(h).cuda() for h in hosts]   # stepped by the workspace variant
    ga = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
    gb = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
    ws = torch.empty(lst.lst_workspace_bytes(), dtype=torch.uint8, device="cuda")
    skip = [0, 0, 0, 1, 0][: L.n_layers]
    stream = torch.cuda.current_stream().cuda_stream
    refs = [h.copy() for h in hosts]
    for call, base_t in enumerate((10, 11)):
        steps = [base_t + 3 * i for i in range(L.n_layers)]
        hp, _ = hparams_for(workload, base_t)
        lst.lst_adamw_step_ex_noalloc(L.handle, [x.data_ptr() for x in a], hp, block_steps=steps, skip=skip,
                                      grad_sq=ga.data_ptr(), stream=stream)
        lst.lst_adamw_step_ex(L.handle, [x.data_ptr() for x in b], hp,
                              lst.step_options(block_steps=steps, skip=skip, grad_sq=gb.data_ptr(),
                                               workspace=ws.data_ptr()), stream)
        torch.cuda.synchronize()
        g_a, g_b = ga.cpu().numpy(), gb.cpu().numpy()
        for i in range(L.n_layers):
            got = L.numpy_views(i, a[i].cpu().numpy())
            exp = L.numpy_views(i, b[i].cpu().numpy())
            compare(fmt, got, exp)
            assert np.array_equal(got["G"], exp["G"])
            if skip[i]:
                assert np.array_equal(a[i].cpu().numpy(), hosts[i]) and g_a[i] == -1.0
                continue
            assert abs(g_a[i] - g_b[i]) <= GSQ_REL * g_b[i], (call, i, g_a[i], g_b[i])
            # and both against the oracle
            G = L.numpy_views(i, refs[i])["G"]
            assert abs(g_a[i] - oracle.grad_sq(G)) <= GSQ_REL * oracle.grad_sq(G)
            oracle.step(fmt, L.numpy_views(i, refs[i]), hparams_for(workload, steps[i])[1])
            compare(fmt, got, L.numpy_views(i, refs[i]))


def test_noalloc_more_blocks_than_one_launch_holds():
    """300 ragged blocks (three update launches, each followed by its reduce
    launch) share the one scratch array in stream order: results and sums of
    g^2 match the workspace variant and the oracle, on two calls in a row."""
    L = Layout([(f"t{i}", (1000 + 37 * i,), i) for i in range(300)], "L12")
    hosts = [np.empty(L.block_bytes(i), np.uint8) for i in range(L.n_layers)]
    for i in range(L.n_layers):
        fill_host_block(L, i, hosts[i], "many", 3)
    a = [torch.from_numpy(h).cuda() for h in hosts]
    b = [torch.from_numpy(h).cuda() for h in hosts]
    ga = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
    gb = torch.full((L.n_layers,), -1.0, dtype=torch.float64, device="cuda")
    ws = torch.empty(lst.lst_workspace_bytes(), dtype=torch.uint8, device="cuda")
    skip = [1 if i % 97 == 5 else 0 for i in range(L.n_layers)]
    refs = [h.copy() for h in hosts]
    stream = torch.cuda.current_stream().cuda_stream
    for t in (3, 4):
        hp, ohp = hparams_for("many", t)
        lst.lst_adamw_step_ex_noalloc(L.handle, [x.data_ptr() for x in a], hp, skip=skip, grad_sq=ga.data_ptr(),
                                      stream=stream)
        lst.lst_adamw_step_ex(L.handle, [x.data_ptr() for x in b], hp,
                              lst.step_options(skip=skip, grad_sq=gb.data_ptr(), workspace=ws.data_ptr()), stream)
        torch.cuda.synchronize()
        g_a, g_b = ga.cpu().numpy(), gb.cpu().numpy()
        for i in range(L.n_layers):
            got = a[i].cpu().numpy()
            assert np.array_equal(got, b[i].cpu().numpy()), (t, i)
            if skip[i]:
                assert np.array_equal(got, hosts[i]) and g_a[i] == -1.0
                continue
            exp_sq = oracle.grad_sq(L.numpy_views(i, refs[i])["G"])
            assert abs(g_a[i] - g_b[i]) <= GSQ_REL * g_b[i] and abs(g_a[i] - exp_sq) <= GSQ_REL * exp_sq, (t, i)
            oracle.step("L12", L.numpy_views(i, refs[i]), ohp)
            assert np.array_equal(got, refs[i]), (t, i)


def test_noalloc_call_that_fails_validation_touches_nothing():
    """A refused call (a block step below 1, a misaligned grad_sq, bad
    hyperparameters) leaves the blocks and the sums exactly as they were."""
    L = Layout([(f"t{i}", (4096 + i,), i) for i in range(3)], "L16M")
    hosts = [np.empty(L.block_bytes(i), np.uint8) for i in range(L.n_layers)]
    for i in range(L.n_layers):
        fill_host_block(L, i, hosts[i], "refuse", 5)
    dev = [torch.from_numpy(h).cuda() for h in hosts]
    gsq = torch.full((L.n_layers + 1,), 1234.5, dtype=torch.float64, device="cuda")
    ptrs = [d.data_ptr() for d in dev]
    hp, _ = hparams_for("refuse", 5)
    cases = [
        (dict(block_steps=[5, 0, 5], grad_sq=gsq.data_ptr()), lst.LST_ERR_INVALID_ARG),
        (dict(grad_sq=gsq.data_ptr() + 4), lst.LST_ERR_ALIGNMENT),
    ]
    for kw, status in cases:
        with pytest.raises(lst.LstError) as e:
            lst.lst_adamw_step_ex_noalloc(L.handle, ptrs, hp, **kw)
        assert e.value.status == status
    bad = lst.adamw_hparams(step=5, beta1=1.0)
    with pytest.raises(lst.LstError) as e:
        lst.lst_adamw_step_ex_noalloc(L.handle, ptrs, bad, grad_sq=gsq.data_ptr())
    assert e.value.status == lst.LST_ERR_INVALID_ARG
    torch.cuda.synchronize()
    for i in range(L.n_layers):
        assert np.array_equal(dev[i].cpu().numpy(), hosts[i]), i
    assert np.all(gsq.cpu().numpy() == 1234.5)
