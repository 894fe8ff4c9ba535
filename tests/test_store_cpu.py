"""The file-backed block store without a GPU: format, persistence, atomic
commit under a simulated crash, layout checks (host-only calls)."""

import os

import numpy as np
import pytest

from optimizer_update_gb300 import Layout, lst


def aligned(nbytes, fill=None):
    raw = np.zeros(nbytes + 4096, np.uint8)
    off = (-raw.ctypes.data) % 4096
    a = raw[off:off + nbytes]
    if fill is not None:
        a[:] = fill
    return a


@pytest.fixture
def layout():
    L = Layout([("a", (3000,), 0), ("b", (9,), 1), ("c", (5000,), 2)], "L12")
    yield L
    L.close()


@pytest.fixture(autouse=True)
def _clear_inject():
    lst.lst_test_inject(0, 0)
    yield
    lst.lst_test_inject(0, 0)


def test_create_open_read_back(layout, tmp_path):
    rng = np.random.default_rng(1)
    blocks = [aligned(layout.block_bytes(i)) for i in range(layout.n_layers)]
    for b in blocks:
        b[:] = rng.integers(0, 256, b.size, dtype=np.uint8)
    S = lst.lst_store_create(layout.handle, str(tmp_path), [b.ctypes.data for b in blocks], 7)
    lst.lst_store_close(S)
    files = sorted(os.listdir(tmp_path))
    assert files == [f"block_{i:06d}.lst" for i in range(3)]
    for i in range(3):
        assert os.path.getsize(tmp_path / files[i]) == 4096 + layout.block_bytes(i)
    S = lst.lst_store_open(layout.handle, str(tmp_path))
    for i in range(3):
        assert lst.lst_store_block_step(S, i) == 7
        out = aligned(layout.block_bytes(i))
        lst.lst_store_read(S, i, out.ctypes.data)
        assert np.array_equal(out, blocks[i])
    lst.lst_store_close(S)


def test_zero_blocks_and_write_persists_step(layout, tmp_path):
    S = lst.lst_store_create(layout.handle, str(tmp_path), None, 0)
    out = aligned(layout.block_bytes(1), fill=1)
    lst.lst_store_read(S, 1, out.ctypes.data)
    assert not out.any()
    new = aligned(layout.block_bytes(1), fill=0x3C)
    lst.lst_store_write(S, 1, new.ctypes.data, 5)
    assert lst.lst_store_block_step(S, 1) == 5
    lst.lst_store_close(S)
    S = lst.lst_store_open(layout.handle, str(tmp_path))
    assert [lst.lst_store_block_step(S, i) for i in range(3)] == [0, 5, 0]
    lst.lst_store_read(S, 1, out.ctypes.data)
    assert np.array_equal(out, new)
    lst.lst_store_close(S)


def test_crash_between_flush_and_rename_keeps_the_old_block(layout, tmp_path):
    old = aligned(layout.block_bytes(2), fill=0x11)
    S = lst.lst_store_create(layout.handle, str(tmp_path), [None, None, old.ctypes.data], 3)
    new = aligned(layout.block_bytes(2), fill=0x22)
    lst.lst_test_inject(3, 3)  # the commit of block 2 fails before its rename
    with pytest.raises(lst.LstError) as e:
        lst.lst_store_write(S, 2, new.ctypes.data, 4)
    assert e.value.status == lst.LST_ERR_IO and "injected" in str(e.value)
    assert (tmp_path / "block_000002.lst.new").exists()  # the shadow, fully written
    lst.lst_store_close(S)
    lst.lst_test_inject(0, 0)
    S = lst.lst_store_open(layout.handle, str(tmp_path))  # recovery discards the shadow
    assert not (tmp_path / "block_000002.lst.new").exists()
    assert lst.lst_store_block_step(S, 2) == 3
    out = aligned(layout.block_bytes(2))
    lst.lst_store_read(S, 2, out.ctypes.data)
    assert np.array_equal(out, old)
    lst.lst_store_close(S)


def test_open_rejects_other_layouts_and_damage(layout, tmp_path):
    S = lst.lst_store_create(layout.handle, str(tmp_path), None, 0)
    lst.lst_store_close(S)
    other = Layout([("a", (3000,), 0), ("b", (9,), 1), ("c", (5000,), 2)], "L16M")
    with pytest.raises(lst.LstError) as e:
        lst.lst_store_open(other.handle, str(tmp_path))
    assert e.value.status == lst.LST_ERR_INVALID_ARG
    bigger = Layout([("a", (3000,), 0), ("b", (9,), 1), ("c", (50000,), 2)], "L12")
    with pytest.raises(lst.LstError) as e:
        lst.lst_store_open(bigger.handle, str(tmp_path))
    assert e.value.status == lst.LST_ERR_INVALID_ARG
    with open(tmp_path / "block_000001.lst", "r+b") as f:  # flip a byte of the step counter
        f.seek(48)
        b = f.read(1)
        f.seek(48)
        f.write(bytes([b[0] ^ 1]))
    with pytest.raises(lst.LstError) as e:
        lst.lst_store_open(layout.handle, str(tmp_path))
    assert e.value.status == lst.LST_ERR_IO and "damaged" in str(e.value)
    os.remove(tmp_path / "block_000001.lst")
    with pytest.raises(lst.LstError) as e:
        lst.lst_store_open(layout.handle, str(tmp_path))
    assert e.value.status == lst.LST_ERR_IO
    other.close()
    bigger.close()


def test_argument_checks(layout, tmp_path):
    S = lst.lst_store_create(layout.handle, str(tmp_path), None, 0)
    buf = aligned(layout.max_block_bytes + 64)
    for call in (lambda: lst.lst_store_read(S, 3, buf.ctypes.data),
                 lambda: lst.lst_store_block_step(S, -1)):
        with pytest.raises(lst.LstError) as e:
            call()
        assert e.value.status == lst.LST_ERR_INVALID_ARG
    with pytest.raises(lst.LstError) as e:
        lst.lst_store_read(S, 0, buf.ctypes.data + 64)
    assert e.value.status == lst.LST_ERR_ALIGNMENT
    with pytest.raises(lst.LstError) as e:  # a block two steps behind cannot take step 2
        lst.lst_store_step(S, [buf.ctypes.data] * 3, 4096, 8192, lst.adamw_hparams(step=2), 1000)
    assert e.value.status == lst.LST_ERR_INVALID_ARG
    with pytest.raises(lst.LstError) as e:
        lst.lst_store_step(S, [buf.ctypes.data + 64] * 3, 4096, 8192, lst.adamw_hparams(step=1), 1000)
    assert e.value.status == lst.LST_ERR_ALIGNMENT
    lst.lst_store_close(S)


def test_bench_disk_probe_cleans_up(tmp_path):
    """The bench's disk probe (the bandwidth the store leg is judged against)
    reports positive rates and leaves nothing behind."""
    import bench
    w, r, direct = bench.disk_bandwidth(str(tmp_path), 8 << 20, req=1 << 20)
    assert w > 0 and r > 0 and isinstance(direct, bool)
    assert list(tmp_path.iterdir()) == []
