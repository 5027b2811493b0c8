"""Host-side tests of the C ABI: the library builds for sm_103a, loads, exports
every function include/bdlm.h declares, and rejects bad arguments before any
launch. No compute call is made (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_diffusion_lm_bdlm_gb300 import build

    build.build()
    import block_diffusion_lm_bdlm_gb300 as bd

    return bd.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bdlm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bdlm_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for f in ("bdlm_attn_fwd", "bdlm_attn_bwd", "bdlm_lse_merge"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    import block_diffusion_lm_bdlm_gb300 as bd

    names = declared_functions()
    assert set(names) == set(bd.EXPORTED_SYMBOLS)
    for f in names:
        assert hasattr(lib, f), f


def test_library_is_built_for_sm103a():
    from block_diffusion_lm_bdlm_gb300 import build

    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)
    assert os.path.exists(build.LIB)


def test_status_strings(lib):
    import block_diffusion_lm_bdlm_gb300 as bd

    assert bd.status_string(0) == "BDLM_OK"
    assert bd.status_string(5) == "BDLM_ERR_TIMEOUT"
    assert bd.status_string(99) == "BDLM_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    f = lib.bdlm_attn_fwd_workspace_bytes
    b = lib.bdlm_attn_bwd_workspace_bytes
    assert f(1024, 4, 128, 1) >= 256
    assert f(0, 4, 128, 1) == 0
    assert f(1024, 4, 96, 1) == 0
    L, H, d = 262144, 32, 128
    # the backward keeps D [H, L] and an fp32 dq accumulator [L, H, d]
    assert b(L, H, d, 1) - f(L, H, d, 1) >= L * H * 4 + L * H * d * 4


def _fwd(lib, **kw):
    args = dict(q=16, k=16, v=16, o=16, lse=16, L=256, block=16, heads=2, kv_heads=2, head_dim=64, cu=None,
                n_docs=1, scale=0.0, part=None, ws=256, ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return lib.bdlm_attn_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["L"], args["block"],
                             args["heads"], args["kv_heads"], args["head_dim"], args["cu"], args["n_docs"],
                             args["scale"], args["part"], args["ws"], args["ws_bytes"], args["stream"])


def test_forward_rejects_bad_arguments(lib):
    import block_diffusion_lm_bdlm_gb300 as bd

    INVALID, UNSUP, WS = 1, 2, 3
    assert _fwd(lib, q=None) == INVALID
    assert _fwd(lib, k=17) == INVALID            # misaligned
    assert _fwd(lib, L=255) == INVALID           # odd total length
    p = bd._CPartial(bd.PART_BLOCK_GROUP, 8, 0, 0, 16)
    assert _fwd(lib, L=200, part=ctypes.byref(p)) == INVALID  # n = 100, B = 16: 7 blocks, the last one short
    p = bd._CPartial(bd.PART_BLOCK_GROUP, 7, 0, 0, 16)
    assert _fwd(lib, L=200, part=ctypes.byref(p), ws=None) == WS  # all 7 blocks: accepted up to the workspace
    assert _fwd(lib, heads=3, kv_heads=2) == INVALID
    assert _fwd(lib, head_dim=96) == UNSUP
    assert _fwd(lib, ws=None) == WS
    assert _fwd(lib, ws=272) == WS               # not 256-aligned
    assert _fwd(lib, ws_bytes=16) == WS
    p = bd._CPartial(bd.PART_KEY_WINDOW, 0, 10, 5, None)  # hi <= lo
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID
    p = bd._CPartial(bd.PART_BLOCK_GROUP, 0, 0, 0, None)  # no block list
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID
    p = bd._CPartial(7, 0, 0, 0, None)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID
    p = bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None)
    assert _fwd(lib, part=ctypes.byref(p), cu=256, n_docs=1) == UNSUP  # windows need one sequence
    p = bd._CPartial(bd.PART_BLOCK_GROUP, 1, 0, 0, 16, bd.PART_ACCUMULATE, 0)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID   # only key windows accumulate
    p = bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None, 4, 0)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID   # unknown flag
    p = bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None, 0, 7)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID   # unknown o dtype
    p = bd._CPartial(bd.PART_NONE, 0, 0, 0, None, 0, bd.BDLM_F32)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID   # fp32 o is for partials
    p = bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None, 0, 0, 10, 5)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID   # empty row range
    p = bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None, 0, 0, 0, 300)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID   # rows past the sequence
    p = bd._CPartial(bd.PART_BLOCK_GROUP, 1, 0, 0, 16, 0, 0, 0, 16)
    assert _fwd(lib, part=ctypes.byref(p)) == INVALID   # row ranges are for windows
    assert lib.bdlm_last_launch_count() == 0


def _tasks_call(lib, tasks, n_slots=2, L=256, block=16, heads=4, kv_heads=2, head_dim=128, o_dtype=0,
                ws=256 * 1024, ws_bytes=1 << 30, q=256):
    import block_diffusion_lm_bdlm_gb300 as bd

    arr = bd._task_array(tasks)
    return lib.bdlm_attn_fwd_tasks(q, 512, 768, 1024, 2048, L, block, heads, kv_heads, head_dim, 0.0, arr,
                                   len(tasks), n_slots, o_dtype, ws, ws_bytes, None)


def test_task_list_rejects_bad_tasks(lib):
    import block_diffusion_lm_bdlm_gb300 as bd

    T = bd.Task
    INVALID, UNSUP, WS = 1, 2, 3
    ok = [T(0, 64, 0, 128, 0, 64, 0), T(128, 64, 0, 128, 64, 128, 1)]
    assert _tasks_call(lib, ok, ws=None) == WS          # well-formed up to the missing workspace
    assert _tasks_call(lib, ok, ws_bytes=64) == WS
    assert _tasks_call(lib, ok, q=None) == INVALID
    assert _tasks_call(lib, ok, q=17) == INVALID         # misaligned
    assert _tasks_call(lib, ok, head_dim=96) == UNSUP
    assert _tasks_call(lib, ok, n_slots=1) == INVALID    # slot 1 outside one slot
    assert _tasks_call(lib, ok, o_dtype=5) == INVALID
    assert _tasks_call(lib, []) == INVALID
    bad = [
        T(-1, 64, 0, 128, 0, 64),       # sequence before row 0
        T(200, 64, 0, 128, 0, 64),      # sequence past L
        T(0, 0, 0, 1, 0, 1),            # empty sequence
        T(0, 64, 10, 10, 0, 64),        # empty row range
        T(0, 64, 0, 129, 0, 64),        # rows past 2n
        T(0, 64, 0, 128, 64, 64),       # empty key window
        T(0, 64, 0, 128, 0, 129),       # keys past 2n
        T(0, 64, 0, 128, 0, 64, -1),    # negative slot
    ]
    for t in bad:
        assert _tasks_call(lib, [t]) == INVALID, t
    # two tasks of one slot on overlapping rows; disjoint rows or other slots are fine
    assert _tasks_call(lib, [T(0, 64, 0, 70, 0, 64), T(0, 64, 60, 128, 64, 128)]) == INVALID
    assert _tasks_call(lib, [T(0, 64, 0, 60, 0, 64), T(0, 64, 60, 128, 64, 128)], ws=None) == WS
    assert _tasks_call(lib, [T(0, 64, 0, 70, 0, 64, 0), T(0, 64, 60, 128, 64, 128, 1)], ws=None) == WS
    assert _tasks_call(lib, [T(0, 64, 0, 100, 0, 64), T(64, 32, 0, 64, 0, 64)]) == INVALID  # rows 64..99 of both
    # the reserved field must be 0
    arr = bd._task_array(ok)
    arr[0].reserved = 1
    assert lib.bdlm_attn_fwd_tasks(256, 512, 768, 1024, 2048, 256, 16, 4, 2, 128, 0.0, arr, 2, 2, 0, 256 * 1024,
                                   1 << 30, None) == INVALID
    assert lib.bdlm_last_launch_count() == 0


def test_task_list_backward_rejects_bad_tasks(lib):
    import block_diffusion_lm_bdlm_gb300 as bd

    T = bd.Task
    INVALID, UNSUP, WS = 1, 2, 3

    def call(tasks, n_slots=2, ws=256 * 1024, head_dim=128, dq=4096):
        arr = bd._task_array(tasks)
        return lib.bdlm_attn_bwd_tasks(256, 512, 768, 1024, 2048, 3072, dq, 8192, 16384, 256, 16, 4, 2, head_dim,
                                       0.0, arr, len(tasks), n_slots, ws, 1 << 30, None)

    ok = [T(0, 64, 0, 128, 0, 64, 0), T(0, 64, 0, 128, 64, 128, 0)]   # one slot, disjoint keys, shared rows
    assert call(ok, ws=None) == WS
    assert call(ok, dq=None) == INVALID
    assert call(ok, dq=4100) == INVALID        # misaligned
    assert call(ok, head_dim=96) == UNSUP
    assert call([]) == INVALID
    # two tasks of one slot on overlapping keys; other slots are fine
    assert call([T(0, 64, 0, 64, 0, 70), T(0, 64, 64, 128, 60, 128)]) == INVALID
    assert call([T(0, 64, 0, 64, 0, 70, 0), T(0, 64, 64, 128, 60, 128, 1)], ws=None) == WS
    assert call([T(0, 64, 0, 128, 0, 129)]) == INVALID   # keys past 2n
    assert lib.bdlm_last_launch_count() == 0
    w = bd.bdlm_attn_bwd_tasks_workspace_bytes(ok, 256, 4, 128)
    assert w > bd.bdlm_attn_fwd_tasks_workspace_bytes(ok)  # holds D and the fp32 dq accumulator
    assert w >= 256 * 4 * 128 * 4 + 256 * 4 * 4
    assert bd.bdlm_attn_bwd_tasks_workspace_bytes(ok, 256, 4, 96) == 0


def test_task_list_workspace_size(lib):
    import block_diffusion_lm_bdlm_gb300 as bd

    T = bd.Task
    one = bd.bdlm_attn_fwd_tasks_workspace_bytes([T(0, 1000, 0, 2000, 0, 10)])
    # 2000 query rows split at n = 1000 give 8 + 8 tiles of 128 rows
    many = bd.bdlm_attn_fwd_tasks_workspace_bytes([T(0, 1000, 0, 2000, 0, 10)] * 100)
    assert 0 < one < many
    assert bd.bdlm_attn_fwd_tasks_workspace_bytes([T(0, 10, 5, 5, 0, 10)]) == 0   # empty row range
    assert bd.bdlm_attn_fwd_tasks_workspace_bytes([]) == 0


def test_selftest_rejects_a_missing_workspace(lib):
    assert lib.bdlm_selftest_timeout(None, 256, 1000000, None) == 3   # BDLM_ERR_WORKSPACE
    assert lib.bdlm_selftest_timeout(256, 16, 1000000, None) == 3     # smaller than the header
    assert lib.bdlm_selftest_timeout(272, 256, 1000000, None) == 3    # not 256-byte aligned


def test_backward_and_merge_reject_bad_arguments(lib):
    import block_diffusion_lm_bdlm_gb300 as bd

    def bwd(part, cu=None):
        return lib.bdlm_attn_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 256, 16, 2, 2, 64, cu, 1, 0.0,
                                 ctypes.byref(part), 256, 1 << 20, None)

    # partial backward: the same descriptor checks as the forward
    assert bwd(bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None), cu=256) == 2  # windows need one sequence
    assert bwd(bd._CPartial(bd.PART_KEY_WINDOW, 0, 10, 5, None)) == 1         # hi <= lo
    assert bwd(bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 257, None)) == 1        # past the sequence
    assert bwd(bd._CPartial(bd.PART_BLOCK_GROUP, 0, 0, 0, None)) == 1         # no block list
    assert bwd(bd._CPartial(bd.PART_BLOCK_GROUP, 9, 0, 0, 16)) == 1           # more blocks than n / B
    assert bwd(bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None, bd.PART_ACCUMULATE, 0)) == 1  # forward-only flag
    assert bwd(bd._CPartial(bd.PART_KEY_WINDOW, 0, 0, 64, None, 0, bd.BDLM_F32)) == 1         # bf16 o only
    st = lib.bdlm_attn_bwd(16, 16, 16, 16, 16, None, 16, 16, 16, 256, 16, 2, 2, 64, None, 1, 0.0, None, 256,
                           1 << 20, None)
    assert st == 1
    VP = ctypes.c_void_p
    parts = (VP * 2)(16, 32)
    lses = (VP * 2)(64, 128)
    assert lib.bdlm_lse_merge(parts, lses, 0, 0, 10, 2, 64, 256, 512, None) == 1      # no partials
    assert lib.bdlm_lse_merge(parts, lses, 65, 0, 10, 2, 64, 256, 512, None) == 1     # too many
    assert lib.bdlm_lse_merge(parts, lses, 2, 0, 10, 2, 96, 256, 512, None) == 2      # d = 96
    assert lib.bdlm_lse_merge(parts, lses, 2, 3, 10, 2, 64, 256, 512, None) == 1      # dtype
    assert lib.bdlm_lse_merge(parts, lses, 2, 0, 10, 2, 64, 16, 512, None) == 1       # o aliases a partial
    bad = (VP * 2)(16, 33)
    assert lib.bdlm_lse_merge(bad, lses, 2, 0, 10, 2, 64, 256, 512, None) == 1        # misaligned partial


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import block_diffusion_lm_bdlm_gb300 as bd

    q = torch.zeros(64, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        bd.bdlm_attn_fwd(q, q, q, 16)


def test_binding_derives_the_rows_a_call_reads(lib):
    # the rows of q and k the C ABI reads for each kind of call; the binding
    # refuses tensors of other shapes before anything reaches the GPU
    import torch

    import block_diffusion_lm_bdlm_gb300 as bd

    assert bd._call_rows(512, None, 16) == (512, 512)
    assert bd._call_rows(512, bd.Partial.window(64, 192), 16) == (512, 128)
    assert bd._call_rows(512, bd.Partial.window(64, 192, q_lo=10, q_hi=50), 16) == (40, 128)
    g = bd.Partial.group(torch.tensor([1, 3, 4], dtype=torch.int32))
    assert bd._call_rows(512, g, 16) == (48, 256 + 48)
    with pytest.raises(ValueError):
        bd._call_rows(512, bd.Partial(bd.PART_BLOCK_GROUP), 16)
    q = torch.empty(512, 4, 64)
    bd._shape("q", q, (512, 4, 64))
    with pytest.raises(ValueError, match="q must be shaped"):
        bd._shape("q", q, (511, 4, 64))
    k = torch.empty(128, 2, 64)
    assert bd._check_qkv(q, k, torch.empty(128, 2, 64), 512, bd.Partial.window(64, 192), 16) == (512, 128)
    with pytest.raises(ValueError, match="k must be shaped"):
        bd._check_qkv(q, torch.empty(120, 2, 64), torch.empty(120, 2, 64), 512, bd.Partial.window(64, 192), 16)
    with pytest.raises(ValueError, match="v must be shaped"):
        bd._check_qkv(q, k, torch.empty(128, 2, 32), 512, bd.Partial.window(64, 192), 16)


def test_ctypes_structs_match_the_header(tmp_path):
    # the binding's ctypes mirrors of bdlm_partial and bdlm_task have the C
    # header's size and field offsets (compiled here with the host compiler)
    import shutil
    import subprocess

    import block_diffusion_lm_bdlm_gb300 as bd

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"bdlm_partial": [f for f, _ in bd._CPartial._fields_], "bdlm_task": [f for f, _ in bd._CTask._fields_]}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "bdlm.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'printf("{st} size %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'printf("{st} {f} %zu\\n", offsetof({st}, {f}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for st, cls in (("bdlm_partial", bd._CPartial), ("bdlm_task", bd._CTask)):
        assert got[(st, "size")] == ctypes.sizeof(cls), st
        for f in fields[st]:
            assert got[(st, f)] == getattr(cls, f).offset, (st, f)
    # every field of the C structs is mirrored (no field missing from ctypes)
    hdr = open(os.path.join(ROOT, "include", "bdlm.h")).read()
    for st in fields:
        body = hdr[:hdr.index("} " + st + ";")]
        body = body[body.rindex("typedef struct {"):]
        declared = re.findall(r"\b(\w+)\s*(?:,\s*(\w+)\s*)?;", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
        names = [x for pair in declared for x in pair if x]
        assert sorted(names) == sorted(fields[st]), (st, names)
