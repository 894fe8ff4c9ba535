"""The boundary is plain C: a C99 program includes include/lst.h, links
liblst.so and drives the host-only calls (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

from conftest import ROOT

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "lst.h"

int main(void) {
  /* two blocks: a 4x8 weight and a norm in block 0, a 1000-element tensor in block 1 */
  int32_t ndim[3] = {2, 1, 1};
  int64_t dims[12] = {4, 8, 0, 0, 8, 0, 0, 0, 1000, 0, 0, 0};
  int32_t layer[3] = {0, 0, 1};
  lst_layout* L = NULL;
  lst_status st = lst_layout_create(3, ndim, dims, layer, LST_L16_MIXED, &L);
  if (st != LST_OK) { printf("create: %s\n", lst_status_string(st)); return 1; }
  int64_t n_layers = 0, n_params = 0, max_bytes = 0;
  lst_layout_info(L, &n_layers, &n_params, &max_bytes);
  int64_t bytes = 0, params = 0, padded = 0, off = 0, seg = 0;
  lst_layout_block(L, 1, &bytes, &params, &padded);
  lst_layout_segment(L, 1, LST_FIELD_W, &off, &seg);
  int64_t t_off = 0, t_layer = 0, t_elem = 0;
  lst_layout_tensor(L, 1, LST_FIELD_MASTER, &t_off, &t_layer, &t_elem);
  printf("%lld %lld %lld %lld %lld %lld %lld %lld %lld %lld\n", (long long)n_layers, (long long)n_params,
         (long long)max_bytes, (long long)bytes, (long long)params, (long long)padded, (long long)off,
         (long long)seg, (long long)t_off, (long long)t_elem);
  /* a bad step counter is refused before any CUDA call */
  lst_adamw_hparams hp = {1e-4f, 0.9f, 0.999f, 1e-8f, 0.01f, 0};
  void* blocks[2] = {0, 0};
  st = lst_adamw_step(L, blocks, &hp, NULL);
  printf("%d %s | %s\n", (int)st, lst_status_string(st), lst_last_error());
  /* streamed-step settings: sub-chunk size and copy mode per direction */
  int ok = lst_layout_set_stream_chunk(L, 4096) == LST_OK &&
           lst_layout_set_stream_copy(L, LST_COPY_SM, LST_COPY_ENGINE) == LST_OK &&
           lst_layout_set_stream_copy(L, LST_COPY_AUTO, LST_COPY_AUTO) == LST_OK &&
           lst_layout_set_stream_copy(L, 3, LST_COPY_ENGINE) == LST_ERR_INVALID_ARG;
  lst_copy_choice cc;
  ok = ok && lst_stream_copy_choice(L, 0, &cc) == LST_OK && cc.measured == 0 && cc.kernel_in_chunks == 0 &&
       lst_stream_copy_choice(L, 99, &cc) == LST_ERR_INVALID_ARG;
  printf("%d\n", ok);
  lst_layout_destroy(L);
  return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    from optimizer_update_gb300 import lst
    if not os.path.exists(lst.LIB_PATH):
        from optimizer_update_gb300 import build
        build.build()
    return os.path.dirname(lst.LIB_PATH)


def test_c99_program_uses_the_abi(libdir, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_lst.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_lst"
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-llst", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    nums = [int(x) for x in out[0].split()]
    # block 0: 32 + 8 params, block 1: 1000 params; each padded to 2048 elements
    assert nums[:3] == [2, 1040, 16 * 2048]
    assert nums[3:6] == [16 * 2048, 1000, 2048]
    assert nums[6:8] == [14 * 2048, 2 * 2048]        # W is the last segment of the mixed layout
    # tensor 1 (the norm) sits after the 32-element weight in block 0: its
    # master data starts after the bf16 G segment, 32 fp32 elements in
    assert nums[8:10] == [2 * 2048 + 32 * 4, 32]
    assert out[1].startswith("1 invalid argument")
    assert out[2] == "1"


STRUCT_PROGRAM = r"""
#include <stddef.h>
#include <stdio.h>
#include "lst.h"
#define F(T, f) printf(#T " " #f " %zu %zu\n", offsetof(T, f), sizeof(((T*)0)->f))
int main(void) {
  printf("lst_adamw_hparams - %zu 0\n", sizeof(lst_adamw_hparams));
  F(lst_adamw_hparams, lr); F(lst_adamw_hparams, beta1); F(lst_adamw_hparams, beta2);
  F(lst_adamw_hparams, eps); F(lst_adamw_hparams, weight_decay); F(lst_adamw_hparams, step);
  printf("lst_step_options - %zu 0\n", sizeof(lst_step_options));
  F(lst_step_options, block_steps); F(lst_step_options, skip); F(lst_step_options, grad_sq);
  F(lst_step_options, workspace);
  printf("lst_copy_choice - %zu 0\n", sizeof(lst_copy_choice));
  F(lst_copy_choice, measured); F(lst_copy_choice, chunks); F(lst_copy_choice, kernel_in_chunks);
  F(lst_copy_choice, kernel_out_chunks); F(lst_copy_choice, engine_h2d_gbs_min);
  F(lst_copy_choice, engine_h2d_gbs_max); F(lst_copy_choice, engine_d2h_gbs_min);
  F(lst_copy_choice, engine_d2h_gbs_max);
  printf("lst_stream_stats - %zu 0\n", sizeof(lst_stream_stats));
  F(lst_stream_stats, steps_completed); F(lst_stream_stats, h2d_bytes); F(lst_stream_stats, d2h_bytes);
  F(lst_stream_stats, chunks); F(lst_stream_stats, kernel_in_chunks); F(lst_stream_stats, kernel_out_chunks);
  F(lst_stream_stats, timed); F(lst_stream_stats, wall_ms); F(lst_stream_stats, h2d_busy_ms);
  F(lst_stream_stats, d2h_busy_ms);
  return 0;
}
"""


def test_c_structs_match_the_binding(tmp_path):
    """Every public struct of include/lst.h has the size, field offsets and
    field sizes that the ctypes binding declares."""
    import ctypes
    from optimizer_update_gb300 import lst
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "structs.c"
    src.write_text(STRUCT_PROGRAM)
    exe = tmp_path / "structs"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    seen = set()
    for line in filter(None, lines):
        name, field, off, size = line.split()
        T = getattr(lst, name)
        if field == "-":
            assert ctypes.sizeof(T) == int(off), name
            continue
        d = getattr(T, field)
        assert (d.offset, d.size) == (int(off), int(size)), (name, field)
        seen.add((name, field))
    for name in ("lst_adamw_hparams", "lst_step_options", "lst_copy_choice", "lst_stream_stats"):
        fields = {f for f, _ in getattr(lst, name)._fields_ if not f.endswith("_")}
        assert fields == {f for n, f in seen if n == name}, name
