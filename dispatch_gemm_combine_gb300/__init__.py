"""GB300 (sm_103a) MoE expert layer: dispatch -> grouped expert FFN -> combine.

Thin ctypes binding of libmoe_gb300.so (declared in include/moe.h).  Every
step of the layer runs in the library's CUDA kernels; this module only
marshals arguments.  PyTorch is used for device memory and streams.  There
is no CPU fallback: if the library is missing or the GPU is not an sm_103
part, calls raise.

Low-level names mirror the C ABI (moe_plan, moe_ffn_fwd, moe_ffn_bwd, ...)
and take raw integers for pointers.  The helpers below them (Shape,
alloc_plan, workspace, plan, ffn_fwd, ffn_bwd) take torch tensors.
"""

import ctypes
import os

__all__ = [
    "MOE_OK", "MOE_ACT_SWIGLU", "MOE_ACT_CLAMPED_GLU", "MOE_BF16", "MOE_FP32", "MoeShape",
    "MoePlan", "MoeBias", "MoeError", "lib", "library_path", "moe_workspace_size", "moe_saved_size",
    "moe_plan", "moe_ffn_fwd", "moe_ffn_bwd", "moe_get_device_error", "moe_status_string",
    "moe_set_wait_timeout_ns", "moe_kernel_launch_count", "moe_profile_enable",
    "moe_profile_read", "moe_profile_kernel_name", "Shape", "alloc_plan", "workspace", "plan", "ffn_fwd", "ffn_bwd",
    "bias_struct", "check_device_error", "moe_gather_rows", "moe_combine_rows", "gather_rows",
    "combine_rows",
]

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_BAD_INDEX = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_CUDA = 6
MOE_ACT_SWIGLU = 0
MOE_ACT_CLAMPED_GLU = 1
MOE_GATE_UP_CONCAT = 0
MOE_GATE_UP_INTERLEAVED = 1
MOE_BF16 = 0
MOE_FP32 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmoe_gb300.so")


class MoeShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("act", ctypes.c_int32),
                ("clamp_limit", ctypes.c_float), ("alpha", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("gate_up_layout", ctypes.c_int32),
                ("out_fp32", ctypes.c_int32)]


class MoePlan(ctypes.Structure):
    _fields_ = [("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("inv", ctypes.c_void_p)]


class MoeBias(ctypes.Structure):
    """moe_bias_t: optional per-expert biases and their gradient outputs."""
    _fields_ = [("b_gate_up", ctypes.c_void_p), ("b_down", ctypes.c_void_p),
                ("db_gate_up", ctypes.c_void_p), ("db_down", ctypes.c_void_p)]


class MoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, moe_status_string(status), status))


_lib = None


def lib():
    """Load libmoe_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError("libmoe_gb300.so is not built (run dispatch_gemm_combine_gb300._build"
                           ".build() or __graft_entry__.build())")
    L = ctypes.CDLL(library_path)
    P = ctypes.c_void_p
    S = ctypes.POINTER(MoeShape)
    PL = ctypes.POINTER(MoePlan)
    L.moe_workspace_size.argtypes = [S, ctypes.c_int]
    L.moe_workspace_size.restype = ctypes.c_size_t
    L.moe_saved_size.argtypes = [S]
    L.moe_saved_size.restype = ctypes.c_size_t
    L.moe_plan.argtypes = [S, P, PL, P, ctypes.c_size_t, P]
    L.moe_plan.restype = ctypes.c_int
    L.moe_route.argtypes = [S, P, P, P, PL, P, ctypes.c_size_t, P]
    L.moe_route.restype = ctypes.c_int
    B = ctypes.POINTER(MoeBias)
    L.moe_ffn_fwd.argtypes = [S, P, P, P, P, P, B, PL, P, P, P, ctypes.c_size_t, P]
    L.moe_ffn_fwd.restype = ctypes.c_int
    L.moe_ffn_bwd.argtypes = [S, P, P, P, P, P, P, B, PL, P, P, P, P, P, P, ctypes.c_size_t, P]
    L.moe_ffn_bwd.restype = ctypes.c_int
    L.moe_get_device_error.argtypes = [P, P]
    L.moe_get_device_error.restype = ctypes.c_int
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.moe_set_wait_timeout_ns.restype = ctypes.c_uint64
    L.moe_kernel_launch_count.argtypes = []
    L.moe_kernel_launch_count.restype = ctypes.c_uint64
    L.moe_profile_enable.argtypes = [ctypes.c_int]
    L.moe_profile_enable.restype = ctypes.c_int
    L.moe_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_uint64), ctypes.c_int]
    L.moe_profile_read.restype = ctypes.c_int
    L.moe_profile_kernel_name.argtypes = [ctypes.c_int]
    L.moe_profile_kernel_name.restype = ctypes.c_char_p
    L.moe_gather_rows.argtypes = [P, ctypes.c_int64, ctypes.c_int32, P, ctypes.c_int64,
                                  ctypes.c_int64, P, P]
    L.moe_gather_rows.restype = ctypes.c_int
    L.moe_combine_rows.argtypes = [S, P, P, P, ctypes.c_int32, P, P]
    L.moe_combine_rows.restype = ctypes.c_int
    _lib = L
    return L


# ---------------------------------------------------------------- raw C ABI
def moe_workspace_size(shape, which):
    return lib().moe_workspace_size(ctypes.byref(shape), which)


def moe_saved_size(shape):
    return lib().moe_saved_size(ctypes.byref(shape))


def moe_plan(shape, topk_idx, plan, ws, ws_bytes, stream):
    return lib().moe_plan(ctypes.byref(shape), topk_idx, ctypes.byref(plan), ws, ws_bytes, stream)


def _byref(st):
    return ctypes.byref(st) if st is not None else None


def moe_ffn_fwd(shape, x, topk_idx, topk_w, w_gate_up, w_down, bias, plan, y, saved, ws,
                ws_bytes, stream):
    return lib().moe_ffn_fwd(ctypes.byref(shape), x, topk_idx, topk_w, w_gate_up, w_down,
                             _byref(bias), _byref(plan), y, saved, ws, ws_bytes, stream)


def moe_ffn_bwd(shape, dy, x, topk_idx, topk_w, w_gate_up, w_down, bias, plan, saved, dx,
                d_topk_w, dw_gate_up, dw_down, ws, ws_bytes, stream):
    return lib().moe_ffn_bwd(ctypes.byref(shape), dy, x, topk_idx, topk_w, w_gate_up, w_down,
                             _byref(bias), _byref(plan), saved, dx, d_topk_w, dw_gate_up,
                             dw_down, ws, ws_bytes, stream)


def moe_get_device_error(ws, stream):
    return lib().moe_get_device_error(ws, stream)


def moe_status_string(status):
    return lib().moe_status_string(status).decode()


def moe_set_wait_timeout_ns(ns):
    return lib().moe_set_wait_timeout_ns(ns)


def moe_kernel_launch_count():
    return lib().moe_kernel_launch_count()


def moe_profile_enable(on):
    return lib().moe_profile_enable(1 if on else 0)


def moe_profile_kernel_name(kind):
    n = lib().moe_profile_kernel_name(kind)
    return None if n is None else n.decode()


def moe_profile_read():
    """{kernel kind name: (total ms, launches)} since the last read."""
    n = 32
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_uint64 * n)()
    k = lib().moe_profile_read(ms, cnt, n)
    return {moe_profile_kernel_name(i): (ms[i], cnt[i]) for i in range(min(k, n))}


def moe_gather_rows(index, n, div, src, src_rows, row_bytes, dst, stream):
    return lib().moe_gather_rows(index, n, div, src, src_rows, row_bytes, dst, stream)


def moe_combine_rows(shape, inv, topk_w, src, src_fp32, dst, stream):
    return lib().moe_combine_rows(ctypes.byref(shape), inv, topk_w, src, 1 if src_fp32 else 0,
                                  dst, stream)


def moe_plan_noalloc(shape, topk_idx, plan, stream):
    """moe_plan without a workspace, for callers that cannot allocate device
    memory when they build a plan; its scratch is a fixed array inside the
    library (see include/moe.h for the size limit and the sharing rules)."""
    fn = lib().moe_plan_noalloc
    fn.argtypes = [ctypes.POINTER(MoeShape), ctypes.c_void_p, ctypes.POINTER(MoePlan),
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn(ctypes.byref(shape), topk_idx, ctypes.byref(plan), stream)


# ---------------------------------------------------------------- torch helpers
def Shape(T, H, I, E, k, act=MOE_ACT_SWIGLU, dtype=MOE_BF16, clamp_limit=7.0, alpha=1.702,
          gate_up_layout=0, out_fp32=0):
    return MoeShape(T, H, I, E, k, act, clamp_limit, alpha, dtype, gate_up_layout,
                    1 if out_fp32 else 0)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def alloc_plan(shape, device="cuda"):
    """int32 device tensors for a plan plus the MoePlan struct pointing at them."""
    import torch
    Tk = max(1, shape.T * shape.k)
    t = {"counts": torch.empty(shape.E, dtype=torch.int32, device=device),
         "offsets": torch.empty(shape.E + 1, dtype=torch.int32, device=device),
         "perm": torch.empty(Tk, dtype=torch.int32, device=device),
         "inv": torch.empty(Tk, dtype=torch.int32, device=device)}
    st = MoePlan(t["counts"].data_ptr(), t["offsets"].data_ptr(), t["perm"].data_ptr(),
                 t["inv"].data_ptr())
    return t, st


def workspace(shape, which, device="cuda"):
    """Zero-filled workspace for call kind `which` (0 plan, 1 fwd, 2 bwd, 3 bwd
    without a saved context)."""
    import torch
    n = moe_workspace_size(shape, which)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def saved_buffer(shape, device="cuda"):
    import torch
    return torch.empty(moe_saved_size(shape), dtype=torch.uint8, device=device)


def route(shape, logits, topk_idx, topk_w, plan_struct=None, ws=None, stream=None):
    """Top-k ids and weights of fp32 logits [T,E] (and the plan, given one)."""
    _check(lib().moe_route(ctypes.byref(shape), _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                           ctypes.byref(plan_struct) if plan_struct is not None else None,
                           _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "moe_route")


def bias_struct(b_gate_up=None, b_down=None, db_gate_up=None, db_down=None):
    """MoeBias over torch tensors (None = absent), or None when all are absent."""
    if all(t is None for t in (b_gate_up, b_down, db_gate_up, db_down)):
        return None
    return MoeBias(_ptr(b_gate_up), _ptr(b_down), _ptr(db_gate_up), _ptr(db_down))


def plan(shape, topk_idx, plan_struct, ws, stream=None):
    _check(moe_plan(shape, _ptr(topk_idx), plan_struct, _ptr(ws), ws.numel(), _stream(stream)),
           "moe_plan")


def ffn_fwd(shape, x, topk_idx, topk_w, w_gate_up, w_down, y, ws, plan_struct=None, saved=None,
            stream=None, bias=None):
    """bias: a MoeBias (see bias_struct) or None."""
    _check(moe_ffn_fwd(shape, _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(w_gate_up),
                       _ptr(w_down), bias, plan_struct, _ptr(y), _ptr(saved), _ptr(ws),
                       ws.numel(), _stream(stream)), "moe_ffn_fwd")


def ffn_bwd(shape, dy, x, topk_idx, topk_w, w_gate_up, w_down, plan_struct, saved, dx, d_topk_w,
            dw_gate_up, dw_down, ws, stream=None, bias=None):
    """bias: a MoeBias (see bias_struct; it also names the bias-gradient
    outputs) or None."""
    _check(moe_ffn_bwd(shape, _ptr(dy), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(w_gate_up),
                       _ptr(w_down), bias, plan_struct, _ptr(saved), _ptr(dx), _ptr(d_topk_w),
                       _ptr(dw_gate_up), _ptr(dw_down), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_ffn_bwd")


def gather_rows(index, div, src, dst, stream=None):
    """dst[r] = src[index[r] // div] for every row r of dst (torch tensors on
    the device; src and dst rows of equal byte size, index int32)."""
    n = index.numel()
    row_bytes = dst.element_size() * (dst.numel() // max(1, dst.shape[0])) if dst.dim() else 0
    if dst.shape[0] != n:
        raise ValueError("gather_rows: dst has %d rows for %d indices" % (dst.shape[0], n))
    src_rows = src.shape[0] if src.dim() else 1
    if n and src.element_size() * (src.numel() // max(1, src_rows)) != row_bytes:
        raise ValueError("gather_rows: src and dst rows differ in size")
    _check(moe_gather_rows(_ptr(index), n, div, _ptr(src), src_rows, row_bytes, _ptr(dst),
                           _stream(stream)), "moe_gather_rows")


def combine_rows(shape, inv, src, dst, topk_w=None, stream=None):
    """dst[t] = sum_j (topk_w[t, j] or 1) * src[inv[t*k + j]] (torch tensors;
    src fp32 or the storage dtype, dst as shape.out_fp32 says)."""
    import torch
    _check(moe_combine_rows(shape, _ptr(inv), _ptr(topk_w), _ptr(src), src.dtype == torch.float32,
                            _ptr(dst), _stream(stream)), "moe_combine_rows")


def check_device_error(ws, stream=None):
    """Synchronise and raise MoeError if a kernel recorded a device-side error."""
    _check(moe_get_device_error(_ptr(ws), _stream(stream)), "device")
