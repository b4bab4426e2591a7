"""Python binding of libretention.so: torch tensors in, pointers out.

Only argument marshalling happens here (dtype/shape checks, the per-call
workspace from torch's caching allocator, the current CUDA stream).  Every
step of the computation runs in the library's CUDA kernels.
"""

from __future__ import annotations

import ctypes as C
from typing import Optional

import numpy as np
import torch

from . import _lib
from ._lib import RET_BF16, RET_F32, RetGN, check, load

_DT = {torch.float32: RET_F32, torch.bfloat16: RET_BF16}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")
    return _DT[t.dtype]


def _host_f32(x, n: int, name: str):
    a = np.ascontiguousarray(np.asarray(x.detach().cpu() if torch.is_tensor(x) else x,
                                        dtype=np.float32).reshape(-1))
    if a.shape[0] != n:
        raise ValueError(f"{name} must have {n} values, got {a.shape[0]}")
    return a, a.ctypes.data_as(C.POINTER(C.c_float))


def _dev(t: Optional[torch.Tensor], name: str, dtype=None, shape=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _gn_struct(gn, H: int, d_v: int, device):
    if not gn:
        return None, []
    keep = []
    w = gn.get("weight") if isinstance(gn, dict) else None
    b = gn.get("bias") if isinstance(gn, dict) else None
    eps = float(gn.get("eps", 1e-5)) if isinstance(gn, dict) else 1e-5
    for name, t in (("gn weight", w), ("gn bias", b)):
        if t is not None:
            _dev(t, name, torch.float32)
            if t.numel() != H * d_v:
                raise ValueError(f"{name} must have H*d_v values")
            keep.append(t)
    s = RetGN(1, eps, C.c_void_p(w.data_ptr()) if w is not None else None,
              C.c_void_p(b.data_ptr()) if b is not None else None)
    return C.byref(s), [s] + keep


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]):
    if nbytes == 0:
        return None, 0, None
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        return C.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(), workspace
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return C.c_void_p(ws.data_ptr()), nbytes, ws


def _check_seq(q, k, v):
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k: [B, H, L, d_k]; v: [B, H, L, d_v]")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    return q.shape[0], q.shape[1], q.shape[2], q.shape[3], v.shape[3]


def plan(form: str, in_dtype, B, H, L, d_k, d_v, chunk=None, out_dtype=None, gn=False,
         gamma=None, state_out=False):
    """(path, workspace bytes) the library would use.  path: 1 = tcgen05, 2 = fp32."""
    lib = load()
    idt = _DT[in_dtype]
    odt = _DT[out_dtype or in_dtype]
    gp = None
    if gamma is not None:
        garr, gp = _host_f32(gamma, H, "gamma")
    path, nbytes = C.c_int(0), C.c_size_t(0)
    if form == "chunkwise":
        st = lib.ret_chunkwise_plan(idt, gp, B, H, L, d_k, d_v, chunk, odt, int(bool(gn)),
                                    C.byref(path), C.byref(nbytes))
    elif form == "chunkwise_compact":
        st = lib.ret_chunkwise_plan_compact(idt, gp, B, H, L, d_k, d_v, chunk, odt, int(bool(gn)),
                                            C.byref(path), C.byref(nbytes))
    elif form == "chunkwise_scan":
        st = lib.ret_chunkwise_scan_plan(idt, gp, B, H, L, d_k, d_v, chunk, odt, int(bool(gn)),
                                         C.byref(path), C.byref(nbytes))
    elif form == "parallel":
        st = lib.ret_parallel_plan(idt, gp, B, H, L, d_k, d_v, odt, int(bool(gn)),
                                   int(bool(state_out)), C.byref(path), C.byref(nbytes))
    else:
        raise ValueError(form)
    check(f"ret_{form}_plan", st)
    return path.value, nbytes.value


def chunk_size(in_dtype, H, L, d_k, d_v, gamma=None) -> int:
    """The library's chunk length for this shape: 128 on the tensor-core path,
    else round(√L)."""
    gp = None
    if gamma is not None:
        garr, gp = _host_f32(gamma, H, "gamma")
    b = load().ret_chunk_size(_DT[in_dtype], gp, H, L, d_k, d_v)
    if b < 1:
        raise ValueError("invalid shape for ret_chunk_size")
    return b


def chunkwise(q, k, v, gamma, theta, chunk: Optional[int] = None, pos0: int = 0, state_in=None,
              return_state: bool = True, out=None, out_dtype=None, gn=None, workspace=None,
              stream=None, layout: str = "carry", state_out=None, compact: bool = False):
    """Chunkwise retention.  Returns (out, state_out or None).

    chunk=None takes ret_chunk_size's choice.
    layout="carry" runs ret_chunkwise (state carried across chunks);
    layout="scan" runs ret_chunkwise_scan (chunk-parallel then scan).
    pos0 is one start position, or a sequence of B start positions (one per
    batch row: ret_chunkwise_rowpos, carry layout).
    compact=True allocates only ret_chunkwise_plan_compact's workspace (the
    Θ prologue inside the chunk launch where that mode applies).
    out / state_out / workspace may be given to avoid allocations.
    """
    lib = load()
    B, H, L, d_k, d_v = _check_seq(q, k, v)
    idt = _dtype_code(q)
    if chunk is None:
        chunk = chunk_size(q.dtype, H, L, d_k, d_v, gamma)
    odtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, L, d_v), dtype=odtype, device=q.device)
    odt = _dtype_code(out)
    garr, gp = _host_f32(gamma, H, "gamma")
    tarr, tp = _host_f32(theta, d_k // 2, "theta")
    st_in = _dev(state_in, "state_in", torch.float32, (B, H, d_k, d_v))
    if state_out is None and return_state:
        state_out = torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=q.device)
    gns, keep = _gn_struct(gn, H, d_v, q.device)
    form = "chunkwise_scan" if layout == "scan" else ("chunkwise_compact" if compact else "chunkwise")
    _, nbytes = plan(form, q.dtype, B, H, L, d_k, d_v, chunk, odtype, bool(gn), gamma=garr)
    wsp, wsn, ws = _workspace(nbytes, q.device, workspace)
    if np.ndim(pos0) == 1:   # one start position per batch row
        if layout != "carry":
            raise ValueError("per-row start positions use the carry layout")
        rows = np.ascontiguousarray(np.asarray(pos0, dtype=np.int64))
        if rows.shape != (B,):
            raise ValueError(f"pos0 needs {B} start positions, got {rows.shape}")
        fn = lib.ret_chunkwise_rowpos
        st = fn(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), idt, gp, tp, B, H, L, d_k, d_v,
                rows.ctypes.data_as(C.POINTER(C.c_int64)), int(chunk), st_in,
                _dev(state_out, "state_out"), _dev(out, "out"), odt, gns, wsp, wsn, _stream(stream))
    else:
        fn = lib.ret_chunkwise_scan if layout == "scan" else lib.ret_chunkwise
        st = fn(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), idt, gp, tp, B, H, L, d_k, d_v, int(pos0),
                int(chunk), st_in, _dev(state_out, "state_out"), _dev(out, "out"), odt, gns, wsp, wsn,
                _stream(stream))
    check(fn.__name__, st)
    return out, state_out


def backward_plan(in_dtype, B, H, L, d_k, d_v, chunk, gamma=None):
    """(path, workspace bytes) of the gradient pass (1 = tcgen05, 2 = fp32 kernels)."""
    lib = load()
    gp = None
    if gamma is not None:
        garr, gp = _host_f32(gamma, H, "gamma")
    path, nbytes = C.c_int(0), C.c_size_t(0)
    check("ret_chunkwise_backward_plan",
          lib.ret_chunkwise_backward_plan(_DT[in_dtype], gp, B, H, L, d_k, d_v, int(chunk),
                                          C.byref(path), C.byref(nbytes)))
    return path.value, nbytes.value


def chunkwise_backward(q, k, v, d_out, gamma, theta, chunk: int, pos0: int = 0, state_in=None,
                       d_state_out=None, return_d_state_in: bool = True, grad_dtype=None,
                       grads=None, d_state_in=None, workspace=None, stream=None):
    """Gradients of chunkwise retention (no GroupNorm) for upstream gradients
    d_out [B, H, L, d_v] (dtype of q) and d_state_out [B, H, d_k, d_v] fp32
    (None = 0).  Returns (dq, dk, dv, d_state_in or None).  grads may be a
    (dq, dk, dv) tuple of preallocated outputs; d_state_in a preallocated
    fp32 state (it may be state_in or d_state_out itself)."""
    lib = load()
    B, H, L, d_k, d_v = _check_seq(q, k, v)
    idt = _dtype_code(q)
    _dev(d_out, "d_out", q.dtype, (B, H, L, d_v))
    gdtype = grad_dtype or q.dtype
    if grads is None:
        grads = (torch.empty((B, H, L, d_k), dtype=gdtype, device=q.device),
                 torch.empty((B, H, L, d_k), dtype=gdtype, device=q.device),
                 torch.empty((B, H, L, d_v), dtype=gdtype, device=q.device))
    dq, dk, dv = grads
    gdt = _dtype_code(dq)
    for name, t, shp in (("dq", dq, (B, H, L, d_k)), ("dk", dk, (B, H, L, d_k)), ("dv", dv, (B, H, L, d_v))):
        _dev(t, name, dq.dtype, shp)
    garr, gp = _host_f32(gamma, H, "gamma")
    tarr, tp = _host_f32(theta, d_k // 2, "theta")
    sshape = (B, H, d_k, d_v)
    if d_state_in is None and return_d_state_in:
        d_state_in = torch.empty(sshape, dtype=torch.float32, device=q.device)
    _, nbytes = backward_plan(q.dtype, B, H, L, d_k, d_v, chunk, gamma=garr)
    wsp, wsn, ws = _workspace(nbytes, q.device, workspace)
    st = lib.ret_chunkwise_backward(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(d_out, "d_out"), idt, gp, tp, B, H, L, d_k,
        d_v, int(pos0), int(chunk), _dev(state_in, "state_in", torch.float32, sshape),
        _dev(d_state_out, "d_state_out", torch.float32, sshape), _dev(dq, "dq"), _dev(dk, "dk"),
        _dev(dv, "dv"), gdt, _dev(d_state_in, "d_state_in", torch.float32, sshape), wsp, wsn, _stream(stream))
    check("ret_chunkwise_backward", st)
    return dq, dk, dv, d_state_in


def param_grads(q, k, v, d_out, out, dq, dk, dv, gamma, theta, pos0: int = 0, state_in=None,
                d_state_out=None, want_gamma: bool = True, want_theta: bool = True, workspace=None,
                stream=None):
    """Gradients with respect to γ [H] and θ [d_k/2] (fp32 device tensors;
    None where not wanted), from the forward call's out and the backward
    call's dq, dk, dv for the same inputs and upstream gradients."""
    lib = load()
    B, H, L, d_k, d_v = _check_seq(q, k, v)
    idt = _dtype_code(q)
    _dev(d_out, "d_out", q.dtype, (B, H, L, d_v))
    _dev(out, "out", None, (B, H, L, d_v))
    gdt = _dtype_code(dq)
    for name, t, shp in (("dq", dq, (B, H, L, d_k)), ("dk", dk, (B, H, L, d_k)), ("dv", dv, (B, H, L, d_v))):
        _dev(t, name, dq.dtype, shp)
    garr, gp = _host_f32(gamma, H, "gamma")
    tarr, tp = _host_f32(theta, d_k // 2, "theta")
    sshape = (B, H, d_k, d_v)
    d_gamma = torch.empty(H, dtype=torch.float32, device=q.device) if want_gamma else None
    d_theta = torch.empty(d_k // 2, dtype=torch.float32, device=q.device) if want_theta else None
    nb = C.c_size_t(0)
    check("ret_chunkwise_param_grads_plan", lib.ret_chunkwise_param_grads_plan(B, H, L, d_k, d_v, C.byref(nb)))
    wsp, wsn, ws = _workspace(nb.value, q.device, workspace)
    st = lib.ret_chunkwise_param_grads(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(d_out, "d_out"), idt, _dev(out, "out"),
        _dtype_code(out), _dev(dq, "dq"), _dev(dk, "dk"), _dev(dv, "dv"), gdt, gp, tp, B, H, L, d_k, d_v,
        int(pos0), _dev(state_in, "state_in", torch.float32, sshape),
        _dev(d_state_out, "d_state_out", torch.float32, sshape), _dev(d_gamma, "d_gamma"),
        _dev(d_theta, "d_theta"), wsp, wsn, _stream(stream))
    check("ret_chunkwise_param_grads", st)
    return d_gamma, d_theta


def groupnorm(x, eps: float = 1e-5, weight=None, bias=None, out=None, out_dtype=None, stream=None):
    """Per-head GroupNorm of x [B, H, L, d_v] over d_v (out may be x)."""
    lib = load()
    if x.dim() != 4:
        raise ValueError("x: [B, H, L, d_v]")
    B, H, L, d_v = x.shape
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    _dev(out, "out", None, x.shape)
    gns, keep = _gn_struct({"eps": eps, "weight": weight, "bias": bias}, H, d_v, x.device)
    st = lib.ret_groupnorm(_dev(x, "x"), _dtype_code(x), _dev(out, "out"), _dtype_code(out), B, H, L, d_v,
                           gns, _stream(stream))
    check("ret_groupnorm", st)
    return out


def groupnorm_backward(x, d_y, eps: float = 1e-5, weight=None, grad_dtype=None, want_params: bool = True,
                       workspace=None, stream=None):
    """Gradients of ``groupnorm``: (d_x, d_weight, d_bias); the last two are
    fp32 [H, d_v] (None unless want_params)."""
    lib = load()
    if x.dim() != 4:
        raise ValueError("x: [B, H, L, d_v]")
    B, H, L, d_v = x.shape
    _dev(d_y, "d_y", x.dtype, x.shape)
    if weight is not None:
        _dev(weight, "weight", torch.float32)
        if weight.numel() != H * d_v:
            raise ValueError("weight must have H*d_v values")
    d_x = torch.empty(x.shape, dtype=grad_dtype or x.dtype, device=x.device)
    d_w = torch.empty((H, d_v), dtype=torch.float32, device=x.device) if want_params else None
    d_b = torch.empty((H, d_v), dtype=torch.float32, device=x.device) if want_params else None
    nb = C.c_size_t(0)
    check("ret_groupnorm_backward_plan", lib.ret_groupnorm_backward_plan(B, H, L, d_v, C.byref(nb)))
    wsp, wsn, ws = _workspace(nb.value if want_params else 0, x.device, workspace)
    st = lib.ret_groupnorm_backward(_dev(x, "x"), _dev(d_y, "d_y"), _dtype_code(x), _dev(weight, "weight"),
                                    float(eps), B, H, L, d_v, _dev(d_x, "d_x"), _dtype_code(d_x),
                                    _dev(d_w, "d_weight"), _dev(d_b, "d_bias"), wsp, wsn, _stream(stream))
    check("ret_groupnorm_backward", st)
    return d_x, d_w, d_b


def parallel(q, k, v, gamma, theta, pos0: int = 0, state_in=None, return_state: bool = False,
             out=None, out_dtype=None, gn=None, workspace=None, stream=None):
    """Parallel-form retention.  Returns (out, state_out or None)."""
    lib = load()
    B, H, L, d_k, d_v = _check_seq(q, k, v)
    idt = _dtype_code(q)
    odtype = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, H, L, d_v), dtype=odtype, device=q.device)
    odt = _dtype_code(out)
    garr, gp = _host_f32(gamma, H, "gamma")
    tarr, tp = _host_f32(theta, d_k // 2, "theta")
    st_in = _dev(state_in, "state_in", torch.float32, (B, H, d_k, d_v))
    state_out = torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=q.device) if return_state else None
    gns, keep = _gn_struct(gn, H, d_v, q.device)
    _, nbytes = plan("parallel", q.dtype, B, H, L, d_k, d_v, None, odtype, bool(gn), gamma=garr,
                     state_out=return_state)
    wsp, wsn, ws = _workspace(nbytes, q.device, workspace)
    st = lib.ret_parallel(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), idt, gp, tp, B, H, L, d_k, d_v,
                          int(pos0), st_in, _dev(state_out, "state_out"), _dev(out, "out"), odt, gns,
                          wsp, wsn, _stream(stream))
    check("ret_parallel", st)
    return out, state_out


def step(q, k, v, gamma, theta, pos: int, state, out=None, out_dtype=None, gn=None, stream=None):
    """One decode step; updates `state` [B, H, d_k, d_v] in place.  Returns out [B, H, d_v]."""
    lib = load()
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError("q, k: [B, H, d_k]; v: [B, H, d_v]")
    B, H, d_k = q.shape
    d_v = v.shape[2]
    idt = _dtype_code(q)
    if out is None:
        out = torch.empty((B, H, d_v), dtype=out_dtype or q.dtype, device=q.device)
    odt = _dtype_code(out)
    garr, gp = _host_f32(gamma, H, "gamma")
    tarr, tp = _host_f32(theta, d_k // 2, "theta")
    gns, keep = _gn_struct(gn, H, d_v, q.device)
    st = lib.ret_step(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), idt, gp, tp, B, H, d_k, d_v, int(pos),
                      _dev(state, "state", torch.float32, (B, H, d_k, d_v)), _dev(out, "out"), odt,
                      gns, _stream(stream))
    check("ret_step", st)
    return out


def rotate(x, theta, pos0: int = 0, scale: float = 1.0, out_dtype=None, stream=None):
    """The Θ prologue alone: scale · R((pos0+t)θ) x for x [B, H, L, d]."""
    lib = load()
    B, H, L, d = x.shape
    y = torch.empty_like(x, dtype=out_dtype or x.dtype)
    tarr, tp = _host_f32(theta, d // 2, "theta")
    st = lib.ret_rotate(_dev(x, "x"), _dtype_code(x), tp, B, H, L, d, int(pos0), float(scale),
                        _dev(y, "y"), _dtype_code(y), _stream(stream))
    check("ret_rotate", st)
    return y


def decay_row_norm(out, gamma, pos0: int = 0, stream=None):
    """Row-normalised decay variant, in place on out [B, H, L, d_v] (or [B, H, d_v]
    of a decode step at position pos0): row t divided by Σ_{i≤pos0+t} γ^i."""
    lib = load()
    x = out if out.dim() == 4 else out.unsqueeze(2)
    B, H, L, d_v = x.shape
    garr, gp = _host_f32(gamma, H, "gamma")
    st = lib.ret_decay_row_norm(_dev(out, "out"), _dtype_code(out), gp, B, H, L, d_v, int(pos0),
                                _stream(stream))
    check("ret_decay_row_norm", st)
    return out


def matmul(a, w, out_dtype=None, stream=None):
    """C = A·W on the tensor cores: a [M, K], w [K, N] bf16 (N % 256 == 0, K % 64 == 0)."""
    lib = load()
    if a.dim() != 2 or w.dim() != 2 or a.shape[1] != w.shape[0]:
        raise ValueError("a: [M, K], w: [K, N]")
    M, K = a.shape
    N = w.shape[1]
    c = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    st = lib.ret_matmul(_dev(a, "a", torch.bfloat16), _dev(w, "w", torch.bfloat16), _dev(c, "c"),
                        _dtype_code(c), M, N, K, _stream(stream))
    check("ret_matmul", st)
    return c


def msr_block_plan(B, L, D, H, d_k, d_v, D_out, gamma=None) -> int:
    """Workspace bytes of ret_msr_block."""
    lib = load()
    gp = None
    if gamma is not None:
        garr, gp = _host_f32(gamma, H, "gamma")
    nbytes = C.c_size_t(0)
    check("ret_msr_block_plan", lib.ret_msr_block_plan(gp, B, L, D, H, d_k, d_v, D_out, C.byref(nbytes)))
    return nbytes.value


def msr_block(x, w_q, w_k, w_v, w_g, w_o, gamma, theta, pos0: int = 0, state_in=None,
              return_state: bool = True, gn_eps: float = 1e-5, out=None, out_dtype=None,
              workspace=None, stream=None):
    """The MSR block: z = (swish(x·W_G) ⊙ GN(retention(x·W_Q, x·W_K, x·W_V)))·W_O.

    x [B, L, D] bf16; w_q, w_k [D, H, d_k]; w_v, w_g [D, H, d_v]; w_o [H, d_v, D_out]
    (bf16, contiguous).  Returns (z [B, L, D_out], state_out or None)."""
    lib = load()
    if x.dim() != 3 or w_q.dim() != 3 or w_v.dim() != 3 or w_o.dim() != 3:
        raise ValueError("x [B, L, D]; w_q, w_k [D, H, d_k]; w_v, w_g [D, H, d_v]; w_o [H, d_v, D_out]")
    B, L, D = x.shape
    _, H, d_k = w_q.shape
    d_v, D_out = w_v.shape[2], w_o.shape[2]
    for name, t, shp in (("w_k", w_k, (D, H, d_k)), ("w_v", w_v, (D, H, d_v)), ("w_g", w_g, (D, H, d_v)),
                         ("w_o", w_o, (H, d_v, D_out))):
        _dev(t, name, torch.bfloat16, shp)
    if out is None:
        out = torch.empty((B, L, D_out), dtype=out_dtype or torch.bfloat16, device=x.device)
    garr, gp = _host_f32(gamma, H, "gamma")
    tarr, tp = _host_f32(theta, d_k // 2, "theta")
    sshape = (B, H, d_k, d_v)
    state_out = torch.empty(sshape, dtype=torch.float32, device=x.device) if return_state else None
    nbytes = msr_block_plan(B, L, D, H, d_k, d_v, D_out, gamma=garr)
    wsp, wsn, ws = _workspace(nbytes, x.device, workspace)
    st = lib.ret_msr_block(_dev(x, "x", torch.bfloat16), _dev(w_q, "w_q"), _dev(w_k, "w_k"),
                           _dev(w_v, "w_v"), _dev(w_g, "w_g"), _dev(w_o, "w_o"), gp, tp, B, L, D, H,
                           d_k, d_v, D_out, int(pos0),
                           _dev(state_in, "state_in", torch.float32, sshape),
                           _dev(state_out, "state_out"), _dev(out, "out"), _dtype_code(out),
                           float(gn_eps), wsp, wsn, _stream(stream))
    check("ret_msr_block", st)
    return out, state_out


def sync_status(stream=None) -> int:
    """Synchronise and return (and clear) the device status word as a ret_status code."""
    return load().ret_sync_status(_stream(stream))


def selftest_timeout(budget_us: int, stream=None) -> None:
    check("ret_selftest_timeout", load().ret_selftest_timeout(int(budget_us), _stream(stream)))


def force_path(path: int) -> None:
    """0 = automatic, 2 = fp32 kernels only (cross-checks)."""
    check("ret_force_path", load().ret_force_path(int(path)))


def status_string(code: int) -> str:
    return load().ret_status_string(int(code)).decode()
