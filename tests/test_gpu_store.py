"""File-backed block store on GB300: a store step equals the device-resident
step bit for bit, step counters persist, and a step interrupted between a
block's flush and its rename is completed exactly once per block by calling
it again."""

import numpy as np
import pytest

import oracle
from optimizer_update_gb300 import Layout, lst
from synth import shapes

from gpu_util import PinnedBlocks, compare, fill_host_block, hparams_for, oracle_step

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


def _specs():
    s = [(n, sh, l - 1) for (n, sh, l) in shapes.tinyllama_full() if l in (1, 2)]
    return s + [("odd", (4097,), 2), ("tiny", (9,), 3), ("w", (70_001,), 4)]


@pytest.mark.parametrize("fmt,workload", [("L16M", "tinyllama_full_l16m"), ("L12", "tinyllama_layer_l12")])
def test_store_steps_match_device_steps_and_resume_exactly_once(fmt, workload, tmp_path):
    L = Layout(_specs(), fmt)
    L.set_stream_chunk(1 << 20)
    init = PinnedBlocks(L)
    stage = [lst.lst_host_alloc(L.max_block_bytes) for _ in range(3)]
    try:
        for i in range(L.n_layers):
            fill_host_block(L, i, init.arrays[i], workload, 1)
        S = lst.lst_store_create(L.handle, str(tmp_path), init.ptrs, 0)
        dev = [torch.from_numpy(init.arrays[i].copy()).cuda() for i in range(L.n_layers)]
        ref = [init.arrays[i].copy() for i in range(L.n_layers)]
        b0 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        b1 = torch.empty(L.max_block_bytes, dtype=torch.uint8, device="cuda")
        for t in (1, 2, 3):
            hp, ohp = hparams_for(workload, t)
            if t == 3:
                lst.lst_test_inject(3, 3)  # block 2's commit fails after its flush: blocks 0, 1 are at t
                with pytest.raises(lst.LstError) as e:
                    lst.lst_store_step(S, stage, b0.data_ptr(), b1.data_ptr(), hp, 600_000)
                assert e.value.status == lst.LST_ERR_IO
                lst.lst_test_inject(0, 0)
                lst.lst_store_close(S)
                S = lst.lst_store_open(L.handle, str(tmp_path))
                steps = [lst.lst_store_block_step(S, i) for i in range(L.n_layers)]
                assert steps[:2] == [3, 3] and all(x == 2 for x in steps[2:]), steps
            lst.lst_store_step(S, stage, b0.data_ptr(), b1.data_ptr(), hp, 600_000)
            # calling it again does nothing: every block is at t
            lst.lst_store_step(S, stage, b0.data_ptr(), b1.data_ptr(), hp, 600_000)
            lst.lst_adamw_step(L.handle, [d.data_ptr() for d in dev], hp, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            for i in range(L.n_layers):
                oracle_step(L, ref[i], i, ohp)
        out = PinnedBlocks(L)
        try:
            for i in range(L.n_layers):
                assert lst.lst_store_block_step(S, i) == 3
                lst.lst_store_read(S, i, out.ptrs[i])
                assert np.array_equal(out.arrays[i], dev[i].cpu().numpy()), f"block {i}: store differs"
                compare(fmt, L.numpy_views(i, out.arrays[i]), L.numpy_views(i, ref[i]))
        finally:
            out.free()
        lst.lst_store_close(S)
    finally:
        init.free()
        for p in stage:
            lst.lst_host_free(p)
