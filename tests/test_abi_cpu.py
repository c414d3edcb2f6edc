"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/moe.h declares, and its host-side logic (workspace
sizing, argument validation, status strings) behaves without a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from dispatch_gemm_combine_gb300 import _build
    _build.build()
    import dispatch_gemm_combine_gb300 as m
    return m


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_function(L):
    names = _declared_functions()
    assert "moe_ffn_fwd" in names and "moe_plan" in names and "moe_ffn_bwd" in names
    lib = ctypes.CDLL(L.library_path)
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_sizes(L):
    s = L.Shape(8192, 2880, 2880, 128, 4, L.MOE_ACT_CLAMPED_GLU)
    Tk = 8192 * 4
    rows = (Tk + 128 * 127) // 128 * 128
    fwd = L.moe_workspace_size(s, 1)
    bwd = L.moe_workspace_size(s, 2)
    assert fwd >= rows * (2880 + 2880) * 2
    assert bwd >= rows * (2880 * 2 + 2 * 2880 + 2880) * 2
    # saved: the grouped bf16 x rows, then the gate | up pre-activations,
    # fp16 for the clamped GLU with bf16 storage
    assert L.moe_saved_size(s) == rows * 2880 * 2 + rows * 2 * 2880 * 2
    assert L.moe_workspace_size(s, 0) < fwd
    # a backward without the saved context also holds the grouped x rows and
    # the pre-activations it recomputes
    assert L.moe_workspace_size(s, 3) >= bwd + rows * 2880 * 2 + rows * 2 * 2880 * 2
    assert L.moe_workspace_size(s, 4) == 0
    # few tokens: at most Tk experts hold a row; SwiGLU saves fp32
    s2 = L.Shape(3, 64, 64, 256, 2)
    rows2 = (6 + 6 * 127) // 128 * 128
    assert L.moe_saved_size(s2) == rows2 * 64 * 2 + rows2 * 2 * 64 * 4
    # fp32 storage saves fp32 pre-activations for either activation
    s3 = L.Shape(3, 64, 64, 256, 2, L.MOE_ACT_CLAMPED_GLU, L.MOE_FP32)
    assert L.moe_saved_size(s3) == rows2 * 64 * 4 + rows2 * 2 * 64 * 4
    # fp16 only for a clamp limit that fp16 represents exactly (|L| <= 32768)
    for lim in (40000.0, 7.3):
        assert L.moe_saved_size(L.Shape(3, 64, 64, 256, 2, L.MOE_ACT_CLAMPED_GLU,
                                        clamp_limit=lim)) == rows2 * 64 * 2 + rows2 * 2 * 64 * 4
    assert L.moe_saved_size(L.Shape(3, 64, 64, 256, 2, L.MOE_ACT_CLAMPED_GLU,
                                    clamp_limit=10.0)) == rows2 * 64 * 2 + rows2 * 2 * 64 * 2


@pytest.mark.parametrize("bad", [dict(H=100), dict(I=12), dict(k=0), dict(E=2, k=3),
                                 dict(E=2000), dict(k=33, E=64), dict(T=-1)])
def test_invalid_shapes(L, bad):
    kw = dict(T=16, H=64, I=64, E=8, k=2)
    kw.update(bad)
    s = L.Shape(**kw)
    assert L.moe_workspace_size(s, 1) == 0
    assert L.moe_saved_size(s) == 0
    plan = L.MoePlan(1, 1, 1, 1)
    st = L.moe_plan(s, 1, plan, 1, 1 << 30, None)
    assert st == L.MOE_ERR_INVALID_ARG


def test_validation_before_device_access(L):
    s = L.Shape(16, 64, 64, 8, 2)
    # null workspace / pointers are rejected on the host
    assert L.moe_ffn_fwd(s, 16, 16, 16, 16, 16, None, None, 16, None, None, 0, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_ffn_fwd(s, 0, 16, 16, 16, 16, None, None, 16, None, 256, 1 << 30, None) == L.MOE_ERR_INVALID_ARG
    # misaligned tensors
    assert L.moe_ffn_fwd(s, 24, 16, 16, 16, 16, None, None, 16, None, 256, 1 << 30, None) == L.MOE_ERR_INVALID_ARG
    # workspace too small
    assert L.moe_ffn_fwd(s, 16, 16, 16, 16, 16, None, None, 16, None, 256, 8, None) == L.MOE_ERR_WORKSPACE
    # a misaligned bias or bias gradient
    for b in (L.MoeBias(24, None, None, None), L.MoeBias(None, 40, None, None)):
        assert L.moe_ffn_fwd(s, 16, 16, 16, 16, 16, b, None, 16, None, 256, 1 << 30, None) == L.MOE_ERR_INVALID_ARG
    b = L.MoeBias(None, None, 16, 8)
    assert L.moe_ffn_bwd(s, 16, 16, 16, 16, 16, 16, b, L.MoePlan(16, 16, 16, 16), None, 16, 16, 16,
                         16, 256, 1 << 30, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_status_string(L.MOE_ERR_BAD_INDEX) == "expert index out of range"


def test_wait_timeout_setter(L):
    old = L.moe_set_wait_timeout_ns(12345)
    assert L.moe_set_wait_timeout_ns(old) == 12345


def test_product_path_has_no_oracle_dependency():
    pkg = os.path.join(ROOT, "dispatch_gemm_combine_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in txt.replace("oracle-free", ""), f


def test_struct_layouts_match_the_header(L, tmp_path):
    """The binding's ctypes structs have the C layout of include/moe.h (a
    plain C compiler reads the header on its own and reports each field's
    offset and each struct's size)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"moe_shape": L.MoeShape, "moe_plan_t": L.MoePlan, "moe_bias_t": L.MoeBias}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append('printf("%s size %%zu\\n", sizeof(%s));' % (cname, cname))
        for f, _ in py._fields_:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, f, cname, f))
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)
