"""moe_plan_noalloc: the dispatch plan for callers that cannot allocate device
memory when they build it (its scratch is a fixed array in the library).

Called through the C ABI and compared with moe_plan (which uses a caller
workspace) on two calls in a row of different sizes: the plan is integer
work, so the comparison is exact.  Also checks that a problem beyond the
fixed scratch is refused.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import synth
from synth import ACT_SWIGLU, Recipe

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import dispatch_gemm_combine_gb300 as m
    lib = ctypes.CDLL(m.library_path)
    fn = lib.moe_plan_noalloc
    fn.argtypes = [ctypes.POINTER(m.MoeShape), ctypes.c_void_p, ctypes.POINTER(m.MoePlan),
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def test_plan_noalloc_matches_plan_on_two_calls():
    import dispatch_gemm_combine_gb300 as m
    fn = _noalloc_fn()
    stream = torch.cuda.current_stream()
    cases = [(3000, 8, 256, "zipf", 11), (700, 4, 64, "uniform_ids", 12)]
    for T, k, E, routing, seed in cases:
        r = Recipe("t", T=T, H=64, I=64, E=E, k=k, act=ACT_SWIGLU, weight_std="fan_in",
                   routing=routing, seed=seed)
        idx = synth.make_case(r, with_dy=False).topk_idx.cuda()
        shape = m.Shape(T, 64, 64, E, k)
        ref_t, ref_s = m.alloc_plan(shape)
        ws = m.workspace(shape, 0)
        m.plan(shape, idx, ref_s, ws)
        m.check_device_error(ws)
        out_t, out_s = m.alloc_plan(shape)
        for t in out_t.values():
            t.fill_(-7)
        st = fn(ctypes.byref(shape), idx.data_ptr(), ctypes.byref(out_s), stream.cuda_stream)
        assert st == m.MOE_OK, m.moe_status_string(st)
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "perm", "inv"):
            assert torch.equal(out_t[name], ref_t[name]), name
        assert int(out_t["offsets"][E].item()) == T * k


def test_plan_noalloc_refuses_oversized_problem():
    import dispatch_gemm_combine_gb300 as m
    fn = _noalloc_fn()
    shape = m.Shape(40000, 64, 64, 1024, 8)      # ceil(320000/1024) * 1024 ints > 1 MiB scratch
    _, out_s = m.alloc_plan(m.Shape(1, 64, 64, 1024, 8))
    st = fn(ctypes.byref(shape), 16, ctypes.byref(out_s), torch.cuda.current_stream().cuda_stream)
    assert st == m.MOE_ERR_WORKSPACE


def test_plan_noalloc_wrapper_bad_id_and_launch_count():
    """Through the package wrapper: one expert id set to E on the host (an id
    the plan must leave out) is detectable as offsets[E] == T*k - 1, the
    valid ids are counted exactly, and the call's three kernels and one
    memset show in the launch counter."""
    import dispatch_gemm_combine_gb300 as m
    T, k, E = 900, 4, 32
    r = Recipe("t", T=T, H=64, I=64, E=E, k=k, act=ACT_SWIGLU, weight_std="fan_in",
               routing="uniform_ids", seed=31)
    idx_h = synth.make_case(r, with_dy=False).topk_idx.clone()
    idx_h[17, 2] = E
    idx = idx_h.cuda()
    shape = m.Shape(T, 64, 64, E, k)
    out_t, out_s = m.alloc_plan(shape)
    n0 = m.moe_kernel_launch_count()
    st = m.moe_plan_noalloc(shape, idx.data_ptr(), out_s, torch.cuda.current_stream().cuda_stream)
    assert st == m.MOE_OK, m.moe_status_string(st)
    assert m.moe_kernel_launch_count() - n0 == 4
    torch.cuda.synchronize()
    assert int(out_t["offsets"][E].item()) == T * k - 1
    valid = idx_h.reshape(-1).numpy()
    want = np.bincount(valid[valid < E], minlength=E)
    assert np.array_equal(out_t["counts"].cpu().numpy(), want)
