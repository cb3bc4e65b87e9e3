"""Python binding of libwsa.so: GB300 NaDiT-style 3D window attention.

Thin ctypes marshalling over the C ABI declared in ``include/wsa.h``: every
function below converts torch tensors to device pointers, passes the current
CUDA stream and raises on a non-zero status.  All computation happens in the
library's CUDA kernels; there is no CPU path.  Importing this package fails
loudly when the library has not been built (``__graft_entry__.build()`` or
``python shifted_window_attention_gb300/_build.py``).
"""

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libwsa.so")
# The same ABI built with device-side range checks of every plan-table index.
_CHECKED_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libwsa_checked.so")

REGULAR = 0
SHIFTED = 1
BF16 = 0
FP32 = 1

_STATUS = {
    0: "WSA_OK",
    -1: "WSA_ERR_INVALID_ARG",
    -2: "WSA_ERR_UNSUPPORTED",
    -3: "WSA_ERR_CUDA",
    -4: "WSA_ERR_OOM",
    -5: "WSA_ERR_MISMATCH",
    -6: "WSA_ERR_DEVICE_CHECK",
}


class WsaError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = _STATUS.get(status, str(status))


def _load(path=_LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    i, p, f = ctypes.c_int, ctypes.c_void_p, ctypes.c_float
    ip = ctypes.POINTER(ctypes.c_int)
    sigs = {
        "wsa_version": ([], i),
        "wsa_bounds_checked": ([], i),
        "wsa_debug_fail_allocations": ([i], i),
        "wsa_last_error": ([], ctypes.c_char_p),
        "wsa_window_size": ([i] * 7 + [ip] * 3, i),
        "wsa_layout_windows": ([i] * 8 + [ip, i, ip], i),
        "wsa_plan_create": ([i] * 8 + [p, ctypes.POINTER(p)], i),
        "wsa_plan_destroy": ([p], i),
        "wsa_plan_info": ([p] + [ip] * 7, i),
        "wsa_plan_tables": ([p] + [ctypes.POINTER(p)] * 4, i),
        "wsa_attention": ([p, p, p, p, p, i, i, i, i, f, p], i),
        "wsa_transition": ([p, p, p, p, i, i, p], i),
        "wsa_ensure_layout": ([p, p, p, p, i, i, p, ip], i),
        "wsa_plan_device_status": ([p, ip], i),
        "wsa_attention_noalloc": ([i] * 8 + [p, p, p, p, i, i, f, p], i),
        "wsa_noalloc_device_status": ([ip], i),
        "wsa_attention_text_workspace": ([p, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)], i),
        "wsa_attention_text": ([p] + [p] * 8 + [i, i, i, i, i, f, p, ctypes.c_size_t, p], i),
        "wsa_sp_owners": ([i] * 9 + [ip, i, ip], i),
        "wsa_sp_local_rows": ([i] * 10 + [ip, i, ip], i),
        "wsa_sp_plan_a": ([i] * 11 + [ctypes.POINTER(ctypes.c_longlong), ip, i, ip, i, ip, i, ip, ip, ip], i),
        "wsa_sp_crossover": ([i] * 10 + [ctypes.c_double, p], i),
        "wsa_gather_rows": ([p, i, p, p, i, i, i, p], i),
        "wsa_debug_withhold_units": ([i], i),
        "wsa_rope": ([p, p, p, p, p, i, i, i, i, i, i, f, p], i),
        "wsa_sp_plan_b": ([i] * 8 + [ip, i, ip] + [ctypes.POINTER(ctypes.c_longlong)] * 3
                          + [ctypes.POINTER(ctypes.c_double)], i),
        "wsa_rope_text": ([p, p, p, p, i, i, i, i, i, f, p], i),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()
_checked = None


def checked_library():
    """The bounds-checked build (libwsa_checked.so) as a ctypes library with
    the same signatures as `lib`: every plan-table row index is range-checked
    on the device, and an index out of range is reported by
    wsa_plan_device_status instead of addressing memory."""
    global _checked
    if _checked is None:
        _checked = _load(_CHECKED_LIB_PATH)
    return _checked


def _check(status):
    if status != 0:
        raise WsaError(status, lib.wsa_last_error().decode())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def version():
    return lib.wsa_version()


def window_size(T, H, W, nt, nh, nw, max_temporal=30):
    """Host-only: (wt, wh, ww) of the window note's formula."""
    out = [ctypes.c_int() for _ in range(3)]
    _check(lib.wsa_window_size(T, H, W, nt, nh, nw, max_temporal, *[ctypes.byref(o) for o in out]))
    return tuple(o.value for o in out)


def layout_windows(T, H, W, nt, nh, nw, layout, max_temporal=30):
    """Host-only: list of (t0, t1, h0, h1, w0, w1) in enumeration order."""
    n = ctypes.c_int()
    _check(lib.wsa_layout_windows(T, H, W, nt, nh, nw, layout, max_temporal, None, 0, ctypes.byref(n)))
    buf = (ctypes.c_int * (6 * n.value))()
    _check(lib.wsa_layout_windows(T, H, W, nt, nh, nw, layout, max_temporal, buf, n.value, ctypes.byref(n)))
    return [tuple(buf[6 * k:6 * k + 6]) for k in range(n.value)]


class _DeviceArray:
    """Zero-copy view of a library-owned int32 device table (read-only by the
    library's contract; torch does not model the read-only flag)."""

    def __init__(self, ptr, n, owner):
        self._owner = owner  # keeps the plan alive while the view exists
        self.__cuda_array_interface__ = {
            "shape": (n,), "typestr": "<i4", "data": (ptr, False), "version": 3, "strides": None,
        }


class Plan:
    """One layout's window plan on the current CUDA device (wsa_plan_create)."""

    def __init__(self, T, H, W, nt, nh, nw, layout, max_temporal=30, stream=None):
        h = ctypes.c_void_p()
        _check(lib.wsa_plan_create(T, H, W, nt, nh, nw, layout, max_temporal, _stream(stream),
                                   ctypes.byref(h)))
        self._h = h
        self.T, self.H, self.W = T, H, W
        vals = [ctypes.c_int() for _ in range(7)]
        _check(lib.wsa_plan_info(h, *[ctypes.byref(v) for v in vals]))
        (self.num_windows, self.num_tokens, self.max_window_tokens,
         self.wt, self.wh, self.ww, self.layout) = (v.value for v in vals)

    @property
    def handle(self):
        if self._h is None:
            raise WsaError(-1, "plan was destroyed")
        return self._h

    def tables(self):
        """(offsets, dims, ids, pos) as int32 CUDA tensors sharing the plan's memory."""
        ptrs = [ctypes.c_void_p() for _ in range(4)]
        _check(lib.wsa_plan_tables(self.handle, *[ctypes.byref(x) for x in ptrs]))
        sizes = [self.num_windows + 1, 6 * self.num_windows, self.num_tokens, self.num_tokens]
        dev = torch.device("cuda", torch.cuda.current_device())
        return tuple(torch.as_tensor(_DeviceArray(x.value, n, self), device=dev)
                     for x, n in zip(ptrs, sizes))

    def device_status(self):
        """Synchronises; returns 0 or raises WsaError with the recorded device code."""
        code = ctypes.c_int()
        st = lib.wsa_plan_device_status(self.handle, ctypes.byref(code))
        _check(st)
        return code.value

    def destroy(self):
        if self._h is not None:
            _check(lib.wsa_plan_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            if self._h is not None and lib is not None:
                lib.wsa_plan_destroy(self._h)
                self._h = None
        except Exception:
            pass


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise WsaError(-2, f"unsupported dtype {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def attention(plan, q, k, v, out=None, canonical=True, scale=0.0, stream=None):
    """Per-window softmax(Q K^T * scale) V for all heads.

    q, k, v: CUDA tensors [N, heads, head_dim], contiguous, same dtype (bf16 or
    fp32).  canonical=True: row = canonical token id; False: row = packed
    position of ``plan``.  Returns ``out`` (allocated if None)."""
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise WsaError(-1, "q, k, v must be contiguous 3-D CUDA tensors")
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise WsaError(-1, "q, k, v must share shape and dtype")
    if q.shape[0] != plan.num_tokens:
        raise WsaError(-1, f"q has {q.shape[0]} rows, the plan has {plan.num_tokens} tokens")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise WsaError(-1, "out must match q")
    _check(lib.wsa_attention(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), q.shape[1], q.shape[2],
                             _dtype_code(q), 1 if canonical else 0, float(scale), _stream(stream)))
    return out


def attention_text_workspace_bytes(plan, n_text, heads):
    n = ctypes.c_size_t()
    _check(lib.wsa_attention_text_workspace(plan.handle, n_text, heads, 128, BF16, ctypes.byref(n)))
    return n.value


def attention_text(plan, q, k, v, q_txt, k_txt, v_txt, out=None, out_txt=None, canonical=True, scale=0.0,
                   workspace=None, stream=None):
    """Window attention over [video window, replicated text] segments.

    Returns (video output like q, text output like q_txt): the text output is
    the mean over windows of each window's text rows.  bf16, head_dim 128."""
    for t in (q, k, v, q_txt, k_txt, v_txt):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 3 or t.dtype != torch.bfloat16:
            raise WsaError(-1, "tensors must be contiguous 3-D bf16 CUDA tensors")
    if k.shape != q.shape or v.shape != q.shape or q.shape[0] != plan.num_tokens:
        raise WsaError(-1, "q, k, v must be [N, heads, 128] for the plan")
    if k_txt.shape != q_txt.shape or v_txt.shape != q_txt.shape or q_txt.shape[1:] != q.shape[1:]:
        raise WsaError(-1, "text tensors must be [n_text, heads, 128]")
    n_text, heads = q_txt.shape[0], q.shape[1]
    out = torch.empty_like(q) if out is None else out
    out_txt = torch.empty_like(q_txt) if out_txt is None else out_txt
    need = attention_text_workspace_bytes(plan, n_text, heads)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.wsa_attention_text(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(q_txt), _ptr(k_txt),
                                  _ptr(v_txt), _ptr(out_txt), n_text, heads, 128, BF16, 1 if canonical else 0,
                                  float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))
    return out, out_txt


def transition(src, dst, x, out=None, stream=None):
    """Rows of x (packed order of plan ``src``) rearranged into the packed order
    of plan ``dst``: out[p] = x[pos_src[ids_dst[p]]]."""
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
        raise WsaError(-1, "x must be a contiguous 2-D CUDA tensor")
    if x.shape[0] != src.num_tokens:
        raise WsaError(-1, "x row count does not match the plan")
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise WsaError(-1, "out must match x")
    _check(lib.wsa_transition(src.handle, dst.handle, _ptr(x), _ptr(out), x.shape[1], _dtype_code(x),
                              _stream(stream)))
    return out


def ensure_layout(current, required, x, out=None, stream=None):
    """wsa_ensure_layout: the rows of x (packed order of plan ``current``) in
    the packed order of plan ``required``.  Returns x itself when both plans
    describe the same windows (nothing is launched), else ``out`` (allocated
    if None) holding the transitioned rows."""
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
        raise WsaError(-1, "x must be a contiguous 2-D CUDA tensor")
    if x.shape[0] != current.num_tokens:
        raise WsaError(-1, "x row count does not match the plan")
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise WsaError(-1, "out must match x")
    moved = ctypes.c_int()
    _check(lib.wsa_ensure_layout(current.handle, required.handle, _ptr(x), _ptr(out), x.shape[1], _dtype_code(x),
                                 _stream(stream), ctypes.byref(moved)))
    return out if moved.value else x


def _rope_args(q, k, q_out, k_out):
    for t in (q, k):
        if t is not None and (not t.is_cuda or not t.is_contiguous() or t.dim() != 3):
            raise WsaError(-1, "q and k must be contiguous 3-D CUDA tensors")
    if k is not None and (k.shape != q.shape or k.dtype != q.dtype):
        raise WsaError(-1, "q and k must share shape and dtype")
    q_out = torch.empty_like(q) if q_out is None else q_out
    if k is not None:
        k_out = torch.empty_like(k) if k_out is None else k_out
    for o in (q_out, k_out):
        if o is not None and (o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous()):
            raise WsaError(-1, "outputs must match q")
    return q_out, k_out


def rope(plan, q, k=None, q_out=None, k_out=None, canonical=True, text_len=0, rope_dim=None, theta=10000.0,
         stream=None):
    """wsa_rope: window-local 3D RoPE of q (and k) for ``plan``'s windows.
    Pass q_out=q (k_out=k) to rotate in place.  Returns (q_out, k_out)."""
    q_out, k_out = _rope_args(q, k, q_out, k_out)
    rd = q.shape[2] if rope_dim is None else rope_dim
    _check(lib.wsa_rope(plan.handle, _ptr(q), _ptr(k) if k is not None else None, _ptr(q_out),
                        _ptr(k_out) if k_out is not None else None, q.shape[1], q.shape[2], _dtype_code(q),
                        1 if canonical else 0, int(text_len), rd, float(theta), _stream(stream)))
    return q_out, k_out


def rope_text(q_txt, k_txt=None, q_out=None, k_out=None, rope_dim=None, theta=10000.0, stream=None):
    """wsa_rope_text: RoPE of the text rows, token i at (i, i, i)."""
    q_out, k_out = _rope_args(q_txt, k_txt, q_out, k_out)
    rd = q_txt.shape[2] if rope_dim is None else rope_dim
    _check(lib.wsa_rope_text(_ptr(q_txt), _ptr(k_txt) if k_txt is not None else None, _ptr(q_out),
                             _ptr(k_out) if k_out is not None else None, q_txt.shape[0], q_txt.shape[1],
                             q_txt.shape[2], _dtype_code(q_txt), rd, float(theta), _stream(stream)))
    return q_out, k_out


def gather_rows(x, index, out=None, stream=None):
    """wsa_gather_rows: out[i] = x[index[i]] (the pack and unpack steps of
    the Plan A exchange).  x: contiguous 2-D CUDA tensor; index: int32 CUDA
    tensor.  Indices outside [0, len(x)) leave their rows unwritten."""
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
        raise WsaError(-1, "x must be a contiguous 2-D CUDA tensor")
    if not index.is_cuda or index.dtype != torch.int32 or not index.is_contiguous() or index.dim() != 1:
        raise WsaError(-1, "index must be a contiguous 1-D int32 CUDA tensor")
    rows = index.shape[0]
    if out is None:
        out = torch.empty((rows, x.shape[1]), dtype=x.dtype, device=x.device)
    elif out.shape != (rows, x.shape[1]) or out.dtype != x.dtype or not out.is_contiguous():
        raise WsaError(-1, "out must be [len(index), channels] of x's dtype")
    _check(lib.wsa_gather_rows(_ptr(x), x.shape[0], _ptr(index), _ptr(out), rows, x.shape[1], _dtype_code(x),
                               _stream(stream)))
    return out


def debug_withhold_units(launches):
    """wsa_debug_withhold_units: the next `launches` tensor-core attention
    launches hand out no work unit, so every wait of the kernel runs out and
    the plan's error word records the code (a test hook for the failure
    path); 0 turns it off."""
    _check(lib.wsa_debug_withhold_units(int(launches)))


def attention_noalloc(T, H, W, nt, nh, nw, layout, q, k, v, out, canonical=True, scale=0.0,
                      max_temporal=30, stream=None):
    """wsa_attention_noalloc: bf16 window attention of one layout without a
    plan and without any device allocation (for callers that cannot allocate
    device memory).  ``out`` must be provided by the caller."""
    for t in (q, k, v, out):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 3 or t.dtype != torch.bfloat16:
            raise WsaError(-1, "q, k, v, out must be contiguous 3-D bf16 CUDA tensors")
    if k.shape != q.shape or v.shape != q.shape or out.shape != q.shape or q.shape[2] != 128:
        raise WsaError(-1, "q, k, v, out must share the shape [N, heads, 128]")
    _check(lib.wsa_attention_noalloc(T, H, W, nt, nh, nw, layout, max_temporal, _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(out), q.shape[1], 1 if canonical else 0, float(scale),
                                     _stream(stream)))
    return out


def noalloc_device_status():
    """wsa_noalloc_device_status: synchronises; returns 0 or raises WsaError
    with the code the last allocation-free call's kernels recorded."""
    code = ctypes.c_int()
    _check(lib.wsa_noalloc_device_status(ctypes.byref(code)))
    return code.value


__all__ = [
    "REGULAR", "SHIFTED", "BF16", "FP32", "WsaError", "Plan", "attention", "transition", "ensure_layout",
    "window_size", "layout_windows", "version", "lib", "attention_noalloc", "noalloc_device_status",
    "attention_text",
    "attention_text_workspace_bytes", "gather_rows", "rope", "rope_text",
]
