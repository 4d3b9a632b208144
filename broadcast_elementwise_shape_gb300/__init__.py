"""Python binding of the zr C ABI (``include/zr.h``): argument marshalling only.

Every computation runs in the CUDA kernels of ``_build/libzr.so``; this module
turns torch tensors into ``zr_tensor`` descriptors (data pointer, sizes,
element strides), allocates outputs and workspace with torch on the tensors'
device, passes the current torch stream, and raises ``ZrError`` on a non-zero
status.  There is no CPU fallback: if the library is missing or a tensor is
not on a CUDA device, calls raise.

Entry points mirror the C names:

* ``zr_broadcast_shape(shape_a, shape_b) -> tuple``
* ``zr_binary_fwd(op, a, b, out=None) -> out``
* ``zr_binary_bwd(op, grad_out, a, b, want_a=True, want_b=True, ...) -> (grad_a, grad_b)``
* ``zr_sum_to_shape(x, shape, out=None) -> out``

``op`` is one of ``"add" "sub" "mul" "div"`` or the ``ZR_*`` integer codes.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as _LIB_PATH
from .build import build  # noqa: F401  (re-exported for convenience)

ZR_ADD, ZR_SUB, ZR_MUL, ZR_DIV = 0, 1, 2, 3
OPS = {"add": ZR_ADD, "sub": ZR_SUB, "mul": ZR_MUL, "div": ZR_DIV}
MAX_DIMS = 8

_lib = None


class ZrError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().zr_status_string(status).decode()
        super().__init__(f"{where}: {msg} ({status})")
        self.status = status


class ZrTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("ndim", ctypes.c_int32),
                ("sizes", ctypes.POINTER(ctypes.c_int64)),
                ("strides", ctypes.POINTER(ctypes.c_int64))]


class ZrGrad(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("strides", ctypes.POINTER(ctypes.c_int64)),
                ("accumulate", ctypes.c_int32)]


def lib() -> ctypes.CDLL:
    """The loaded ``libzr.so``; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"zr CUDA library not built ({_LIB_PATH}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_LIB_PATH)
        i64p = ctypes.POINTER(ctypes.c_int64)
        vp, c_int, i32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int32
        szp = ctypes.POINTER(ctypes.c_size_t)
        L.zr_broadcast_shape.argtypes = [i32, i64p, i32, i64p, ctypes.POINTER(i32), i64p]
        L.zr_binary_fwd.argtypes = [c_int, ZrTensor, ZrTensor, vp, i64p, vp]
        L.zr_binary_bwd.argtypes = [c_int, ZrTensor, ZrTensor, ZrTensor, vp, vp, vp, szp, vp]
        L.zr_sum_to_shape.argtypes = [ZrTensor, i32, i64p, vp, vp, szp, vp]
        L.zr_binary_bwd_ex.argtypes = [c_int, ZrTensor, ZrTensor, ZrTensor, ZrGrad, ZrGrad, vp, szp,
                                       vp]
        L.zr_chain_fwd.argtypes = [c_int, c_int, ZrTensor, ZrTensor, ZrTensor, vp, i64p, vp]
        L.zr_unary_fwd.argtypes = [c_int, ctypes.c_float, ZrTensor, vp, i64p, vp]
        L.zr_unary_bwd.argtypes = [c_int, ctypes.c_float, ZrTensor, ZrTensor, vp, i64p, vp]
        L.zr_chain_bwd.argtypes = [c_int, c_int, ZrTensor, ZrTensor, ZrTensor, ZrTensor, vp, vp, vp,
                                   vp, szp, vp]
        L.zr_binary_fwd_t.argtypes = [c_int, c_int, ZrTensor, ZrTensor, vp, i64p, vp]
        L.zr_binary_bwd_t.argtypes = [c_int, c_int, ZrTensor, ZrTensor, ZrTensor, vp, vp, vp, szp, vp]
        L.zr_sum_to_shape_t.argtypes = [c_int, ZrTensor, i32, i64p, vp, vp, szp, vp]
        L.zr_unary_fwd_t.argtypes = [c_int, c_int, ctypes.c_float, ZrTensor, vp, i64p, vp]
        L.zr_unary_bwd_t.argtypes = [c_int, c_int, ctypes.c_float, ZrTensor, ZrTensor, vp, i64p, vp]
        L.zr_status_string.argtypes = [c_int]
        L.zr_status_string.restype = ctypes.c_char_p
        for f in ("zr_broadcast_shape", "zr_binary_fwd", "zr_binary_bwd", "zr_sum_to_shape",
                  "zr_chain_fwd", "zr_chain_bwd", "zr_binary_bwd_ex", "zr_unary_fwd", "zr_unary_bwd",
                  "zr_binary_fwd_t", "zr_binary_bwd_t", "zr_sum_to_shape_t", "zr_unary_fwd_t",
                  "zr_unary_bwd_t"):
            getattr(L, f).restype = c_int
        _lib = L
    return _lib


def _i64(seq):
    return (ctypes.c_int64 * max(1, len(seq)))(*[int(v) for v in seq])


def _desc(t, shape=None, need_data=True):
    """zr_tensor for a torch tensor (or for a shape with no data)."""
    if t is None:
        sizes = _i64(shape)
        return ZrTensor(None, len(shape), sizes, None), (sizes,)
    if need_data and t.numel() > 0 and not t.is_cuda:
        raise ValueError("zr operands must be CUDA tensors")
    import torch
    if t.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("zr operands must be float32 or bfloat16")
    sizes, strides = _i64(t.shape), _i64(t.stride())
    ptr = t.data_ptr() if (t.numel() > 0 and need_data) else None
    return ZrTensor(ptr, t.dim(), sizes, strides), (sizes, strides, t)


def _op(op):
    return OPS[op] if isinstance(op, str) else int(op)


def _stream(t):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check(rc, where):
    if rc != 0:
        raise ZrError(rc, where)


def zr_broadcast_shape(shape_a, shape_b):
    n = ctypes.c_int32(0)
    out = (ctypes.c_int64 * MAX_DIMS)()
    _check(lib().zr_broadcast_shape(len(shape_a), _i64(shape_a), len(shape_b), _i64(shape_b),
                                    ctypes.byref(n), out), "zr_broadcast_shape")
    return tuple(out[i] for i in range(n.value))


def zr_binary_fwd(op, a, b, out=None):
    """out = a op b (broadcasting).  ``out`` may be a preallocated (strided)
    tensor of the broadcast shape; otherwise a contiguous one is allocated."""
    import torch
    dt = _dtype_of(a, b)
    shape = zr_broadcast_shape(a.shape, b.shape)
    if out is None:
        out = torch.empty(shape, dtype=a.dtype, device=a.device)
    elif tuple(out.shape) != shape:
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {shape}")
    _dtype_of(a, out)
    da, ka = _desc(a)
    db, kb = _desc(b)
    ost = _i64(out.stride())
    rc = lib().zr_binary_fwd_t(dt, _op(op), da, db, out.data_ptr() if out.numel() else None, ost,
                               _stream(out))
    _check(rc, "zr_binary_fwd")
    return out


ZR_F32, ZR_BF16 = 0, 1


def _float32_only(where, *ts):
    """The chain and gradient-layout entry points take float32 only."""
    import torch
    for t in ts:
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{where} takes float32 tensors (got {t.dtype})")


def _dtype_of(*ts):
    """The zr_dtype of tensors that must share one element type."""
    import torch
    dts = {t.dtype for t in ts if t is not None}
    if len(dts) > 1:
        raise TypeError(f"operands mix element types {sorted(map(str, dts))}")
    dt = dts.pop() if dts else torch.float32
    if dt == torch.float32:
        return ZR_F32
    if dt == torch.bfloat16:
        return ZR_BF16
    raise TypeError("zr operands must be float32 or bfloat16")


def _workspace(nbytes, device):
    import torch
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def zr_binary_bwd(op, grad_out, a, b, want_a=True, want_b=True, grad_a=None, grad_b=None,
                  shape_a=None, shape_b=None, workspace=None):
    """(grad_a, grad_b) of out = a op b given grad_out.  ``a``/``b`` may be
    None (with ``shape_a``/``shape_b``) when the op does not read them."""
    import torch
    opc = _op(op)
    dt = _dtype_of(grad_out, a, b, grad_a, grad_b)
    sa = tuple(a.shape) if a is not None else tuple(shape_a)
    sb = tuple(b.shape) if b is not None else tuple(shape_b)
    dev = grad_out.device
    if want_a and grad_a is None:
        grad_a = torch.empty(sa, dtype=grad_out.dtype, device=dev)
    if want_b and grad_b is None:
        grad_b = torch.empty(sb, dtype=grad_out.dtype, device=dev)
    dg, kg = _desc(grad_out)
    da, ka = _desc(a, sa)
    db, kb = _desc(b, sb)
    pa = grad_a.data_ptr() if (grad_a is not None and grad_a.numel()) else None
    pb = grad_b.data_ptr() if (grad_b is not None and grad_b.numel()) else None
    if grad_a is not None and grad_a.numel() == 0:
        pa = None
    if grad_b is not None and grad_b.numel() == 0:
        pb = None
    nbytes = ctypes.c_size_t(0)
    _check(lib().zr_binary_bwd_t(dt, opc, dg, da, db, pa, pb, None, ctypes.byref(nbytes), None),
           "zr_binary_bwd (workspace query)")
    if workspace is None or workspace.numel() < nbytes.value:
        workspace = _workspace(nbytes.value, dev)
    nbytes = ctypes.c_size_t(workspace.numel())
    rc = lib().zr_binary_bwd_t(dt, opc, dg, da, db, pa, pb, workspace.data_ptr(),
                               ctypes.byref(nbytes), _stream(grad_out))
    _check(rc, "zr_binary_bwd")
    return grad_a, grad_b


def zr_sum_to_shape(x, shape, out=None, workspace=None):
    """Sum x down to ``shape`` (which must broadcast to x's shape)."""
    import torch
    shape = tuple(int(s) for s in shape)
    if out is None:
        out = torch.empty(shape, dtype=x.dtype, device=x.device)
    dt = _dtype_of(x, out)
    dx, kx = _desc(x)
    so = _i64(shape)
    po = out.data_ptr() if out.numel() else None
    nbytes = ctypes.c_size_t(0)
    _check(lib().zr_sum_to_shape_t(dt, dx, len(shape), so, po, None, ctypes.byref(nbytes), None),
           "zr_sum_to_shape (workspace query)")
    if workspace is None or workspace.numel() < nbytes.value:
        workspace = _workspace(nbytes.value, x.device)
    nbytes = ctypes.c_size_t(workspace.numel())
    rc = lib().zr_sum_to_shape_t(dt, dx, len(shape), so, po, workspace.data_ptr(),
                                 ctypes.byref(nbytes), _stream(x))
    _check(rc, "zr_sum_to_shape")
    return out


def zr_chain_fwd(op1, op2, a, b, c, out=None):
    """out = (a op1 b) op2 c (broadcasting); ``out`` may be a preallocated
    (strided) tensor of the broadcast shape."""
    import torch
    _float32_only("zr_chain_fwd", a, b, c, out)
    shape = zr_broadcast_shape(zr_broadcast_shape(a.shape, b.shape), c.shape)
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=a.device)
    elif tuple(out.shape) != shape:
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {shape}")
    da, ka = _desc(a)
    db, kb = _desc(b)
    dc, kc = _desc(c)
    ost = _i64(out.stride())
    rc = lib().zr_chain_fwd(_op(op1), _op(op2), da, db, dc, out.data_ptr() if out.numel() else None,
                            ost, _stream(out))
    _check(rc, "zr_chain_fwd")
    return out


def zr_chain_bwd(op1, op2, grad_out, a, b, c, want=(True, True, True), grads=(None, None, None),
                 shapes=(None, None, None), workspace=None):
    """(grad_a, grad_b, grad_c) of out = (a op1 b) op2 c given grad_out.  An
    operand may be None (with its shape in ``shapes``) when the requested
    gradients do not read it."""
    import torch
    _float32_only("zr_chain_bwd", grad_out, a, b, c, *grads)
    xs = (a, b, c)
    shp = [tuple(x.shape) if x is not None else tuple(s) for x, s in zip(xs, shapes)]
    dev = grad_out.device
    gs = [g if g is not None else (torch.empty(s, dtype=torch.float32, device=dev) if w else None)
          for g, s, w in zip(grads, shp, want)]
    dg, kg = _desc(grad_out)
    descs = [_desc(x, s) for x, s in zip(xs, shp)]
    ptrs = [g.data_ptr() if (g is not None and g.numel()) else None for g in gs]
    L = lib()
    nbytes = ctypes.c_size_t(0)
    _check(L.zr_chain_bwd(_op(op1), _op(op2), dg, descs[0][0], descs[1][0], descs[2][0], *ptrs,
                          None, ctypes.byref(nbytes), None), "zr_chain_bwd (workspace query)")
    if workspace is None or workspace.numel() < nbytes.value:
        workspace = _workspace(nbytes.value, dev)
    nbytes = ctypes.c_size_t(workspace.numel())
    rc = L.zr_chain_bwd(_op(op1), _op(op2), dg, descs[0][0], descs[1][0], descs[2][0], *ptrs,
                        workspace.data_ptr(), ctypes.byref(nbytes), _stream(grad_out))
    _check(rc, "zr_chain_bwd")
    return tuple(gs)


def _grad(t, acc):
    """zr_grad for a caller's gradient tensor (any strides) or None."""
    if t is None:
        return ZrGrad(None, None, 0), ()
    st = _i64(t.stride())
    return ZrGrad(t.data_ptr() if t.numel() else None, st, 1 if acc else 0), (st, t)


def zr_binary_bwd_ex(op, grad_out, a, b, grad_a=None, grad_b=None, accumulate=(False, False),
                     shape_a=None, shape_b=None, workspace=None):
    """Backward of out = a op b into the caller's gradient tensors, which may
    be strided views; ``accumulate[k]`` adds to what they hold (grad +=
    result) instead of overwriting.  Returns (grad_a, grad_b)."""
    _float32_only("zr_binary_bwd_ex", grad_out, a, b, grad_a, grad_b)
    sa = tuple(a.shape) if a is not None else tuple(shape_a)
    sb = tuple(b.shape) if b is not None else tuple(shape_b)
    for g, s in ((grad_a, sa), (grad_b, sb)):
        if g is not None and tuple(g.shape) != s:
            raise ValueError(f"gradient has shape {tuple(g.shape)}, expected {s}")
    dg, kg = _desc(grad_out)
    da, ka = _desc(a, sa)
    db, kb = _desc(b, sb)
    gga, kga = _grad(grad_a, accumulate[0])
    ggb, kgb = _grad(grad_b, accumulate[1])
    L = lib()
    nbytes = ctypes.c_size_t(0)
    _check(L.zr_binary_bwd_ex(_op(op), dg, da, db, gga, ggb, None, ctypes.byref(nbytes), None),
           "zr_binary_bwd_ex (workspace query)")
    if workspace is None or workspace.numel() < nbytes.value:
        workspace = _workspace(nbytes.value, grad_out.device)
    nbytes = ctypes.c_size_t(workspace.numel())
    rc = L.zr_binary_bwd_ex(_op(op), dg, da, db, gga, ggb, workspace.data_ptr(),
                            ctypes.byref(nbytes), _stream(grad_out))
    _check(rc, "zr_binary_bwd_ex")
    return grad_a, grad_b


UNARY = {"scale": 0, "gelu": 1}


def zr_unary_fwd(op, x, alpha=1.0, out=None):
    """out = op(x) for op in ("scale", "gelu"); ``out`` may be a preallocated
    (strided) tensor of x's shape, or x itself."""
    import torch
    dt = _dtype_of(x, out)
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    dx, kx = _desc(x)
    ost = _i64(out.stride())
    rc = lib().zr_unary_fwd_t(dt, UNARY.get(op, op), float(alpha), dx,
                              out.data_ptr() if out.numel() else None, ost, _stream(out))
    _check(rc, "zr_unary_fwd")
    return out


def zr_unary_bwd(op, grad_out, x, alpha=1.0, grad_x=None):
    """grad_x = grad_out * op'(x); ``x`` may be None for "scale"."""
    import torch
    dt = _dtype_of(grad_out, x, grad_x)
    if grad_x is None:
        grad_x = torch.empty(grad_out.shape, dtype=grad_out.dtype, device=grad_out.device)
    dg, kg = _desc(grad_out)
    dx, kx = _desc(x, tuple(grad_out.shape))
    gst = _i64(grad_x.stride())
    rc = lib().zr_unary_bwd_t(dt, UNARY.get(op, op), float(alpha), dg, dx,
                              grad_x.data_ptr() if grad_x.numel() else None, gst, _stream(grad_out))
    _check(rc, "zr_unary_bwd")
    return grad_x
