"""ret_chunkwise_noalloc: the chunkwise entry point for callers that cannot
allocate device memory (plugins of a host that owns the device memory
budget, latency-critical loops).  It runs the same kernels as ret_chunkwise
with the library's built-in scratch array instead of a caller workspace.

Checked through the C ABI against ret_chunkwise: two calls in a row with
different inputs on each kernel path, and a sequence of calls of different
shapes and paths after the array was filled with NaN by larger problems, so
that a kernel that reads a part of the array it did not write in the same
call shows up.  Plus the size limit.  Collected last on purpose.
"""

import ctypes as C

import numpy as np
import pytest
import torch

import linear_recurrent_sequence_prologue_b300 as R
from linear_recurrent_sequence_prologue_b300 import _lib, build
from linear_recurrent_sequence_prologue_b300.inputs import Workload, make_inputs

from helpers import assert_close

pytestmark = pytest.mark.gpu


def _noalloc(lib, inp, w, pos0, out, state_out, gn=None):
    g = np.ascontiguousarray(inp["gamma"], np.float32)
    t = np.ascontiguousarray(inp["theta"], np.float32)
    fp = lambda a: a.ctypes.data_as(C.POINTER(C.c_float))
    dt = _lib.RET_BF16 if inp["q"].dtype == torch.bfloat16 else _lib.RET_F32
    odt = _lib.RET_BF16 if out.dtype == torch.bfloat16 else _lib.RET_F32
    ptr = lambda x: None if x is None else C.c_void_p(x.data_ptr())
    gns = C.byref(_lib.RetGN(1, gn, None, None)) if gn else None
    st = lib.ret_chunkwise_noalloc(ptr(inp["q"]), ptr(inp["k"]), ptr(inp["v"]), dt, fp(g), fp(t),
                                   w.B, w.H, w.L, w.d_k, w.d_v, pos0, w.chunk,
                                   ptr(inp.get("state_in")), ptr(state_out), ptr(out), odt, gns,
                                   C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _check_against_chunkwise(lib, w, seed, pos0, gn=None):
    inp = make_inputs(w, seed=seed)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    ref_o, ref_s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk,
                               pos0=pos0, state_in=d["state_in"],
                               gn={"eps": gn} if gn else None)
    out = torch.full_like(ref_o, float("nan"))
    s_out = torch.full_like(ref_s, float("nan"))
    assert _noalloc(lib, d, w, pos0, out, s_out, gn) == _lib.RET_OK
    assert R.sync_status() == R.RET_OK
    assert_close(out.double().cpu().numpy(), ref_o.double().cpu().numpy(), w.torch_dtype,
                 f"{w.name} out")
    assert_close(s_out.double().cpu().numpy(), ref_s.double().cpu().numpy(), w.torch_dtype,
                 f"{w.name} state")


@pytest.mark.parametrize("w", [
    Workload("tc", 1, 2, 512, 256, 256, "bf16", 128, 1.0, state_std=0.1),    # tensor-core path
    Workload("tc_ragged", 1, 2, 300, 256, 256, "bf16", 128, 1.0, state_std=0.1),  # short last chunk
    Workload("fp32", 2, 3, 96, 32, 24, "f32", 32, 1.0, state_std=0.1),       # fp32 path
], ids=["tensor_core", "tensor_core_ragged", "fp32"])
def test_noalloc_matches_chunkwise_on_two_calls(w):
    build.build()
    lib = R.load()
    path, need = R.plan("chunkwise", w.torch_dtype, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk)
    assert 0 < need <= _lib.RET_NOALLOC_SCRATCH_BYTES
    for seed in (1, 2):   # second call sees the first call's leftovers in the array
        _check_against_chunkwise(lib, w, seed, 3)


def _poison(lib, w):
    """Run a problem whose inputs are all NaN through the shared array: every
    byte of scratch it uses is left holding NaN (bf16 or fp32)."""
    q = torch.full((w.B, w.H, w.L, w.d_k), float("nan"), dtype=w.torch_dtype, device="cuda")
    v = torch.full((w.B, w.H, w.L, w.d_v), float("nan"), dtype=w.torch_dtype, device="cuda")
    s = torch.full((w.B, w.H, w.d_k, w.d_v), float("nan"), device="cuda")
    inp = {"q": q, "k": q, "v": v, "state_in": s, "gamma": np.full(w.H, 0.97, np.float32),
           "theta": np.ones(w.d_k // 2, np.float32)}
    out = torch.empty_like(v, dtype=torch.float32)
    assert _noalloc(lib, inp, w, 0, out, torch.empty_like(s), 1e-5 if w.groupnorm else None) == _lib.RET_OK
    assert R.sync_status() == R.RET_OK


def test_noalloc_sequence_of_shapes_after_nan_fill():
    """Calls of different shapes and kernel paths share one array: each must
    depend only on what it wrote itself.  The array is first filled with NaN
    by three large problems (tensor cores in both layouts and the fp32 path,
    GroupNorm staging on), then four different problems run back to back."""
    lib = R.load()
    big_tc = Workload("nan_tc", 2, 20, 384, 256, 256, "bf16", 128, 1.0, groupnorm=True)     # carried layout
    big_scan = Workload("nan_scan", 1, 2, 4096, 256, 256, "bf16", 128, 1.0, groupnorm=True)  # chunk-parallel
    big_f32 = Workload("nan_f32", 1, 4, 4096, 64, 64, "f32", 64, 1.0, groupnorm=True)
    for w in (big_tc, big_scan, big_f32):
        need = R.plan("chunkwise", w.torch_dtype, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk,
                      out_dtype=torch.float32, gn=True)[1]
        assert need <= _lib.RET_NOALLOC_SCRATCH_BYTES
        _poison(lib, w)
    seq = [
        (Workload("tc_512", 1, 2, 512, 256, 256, "bf16", 128, 1.0, state_std=0.1), None),
        (Workload("tc_300", 2, 1, 300, 128, 256, "bf16", 128, 1.0, state_std=0.1), None),
        (Workload("f32_gn", 2, 3, 130, 32, 48, "f32", 32, 1.0, state_std=0.1), 1e-5),
        (Workload("tc_gn", 1, 2, 384, 256, 512, "bf16", 128, 1.0, state_std=0.1), 1e-5),
    ]
    for i, (w, gn) in enumerate(seq):
        _check_against_chunkwise(lib, w, 10 + i, 7, gn)


def test_noalloc_runs_the_7b_shape_in_the_compact_mode():
    """The 7B-shape problem needs 268 MB of workspace for the front pass but
    only 25 MB in the compact mode, so it runs from the 32 MiB array; the
    compact mode feeds the same Q″ and K̂′ bits to the same kernels, so the
    result equals ret_chunkwise's (front pass, caller workspace) bit for bit,
    on two calls in a row."""
    lib = R.load()
    w = Workload("msr7b", 2, 16, 8192, 256, 512, "bf16", 128, 1.28, state_std=0.1)
    assert R.plan("chunkwise", w.torch_dtype, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk)[1] > \
        _lib.RET_NOALLOC_SCRATCH_BYTES
    assert R.plan("chunkwise_compact", w.torch_dtype, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk)[1] <= \
        _lib.RET_NOALLOC_SCRATCH_BYTES
    for seed in (3, 4):
        inp = make_inputs(w, seed=seed)
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        ref_o, ref_s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk,
                                   state_in=d["state_in"])
        out = torch.full_like(ref_o, float("nan"))
        s_out = torch.full_like(ref_s, float("nan"))
        assert _noalloc(lib, d, w, 0, out, s_out) == _lib.RET_OK
        assert R.sync_status() == R.RET_OK
        assert torch.equal(out, ref_o) and torch.equal(s_out, ref_s)


def test_noalloc_rejects_problems_beyond_the_array():
    """A problem whose plan needs more scratch than the array holds is
    refused before any launch.  The buffers are real and full-sized, so even a
    launch by mistake would stay in bounds."""
    lib = R.load()
    w = Workload("big", 2, 16, 8192, 256, 512, "f32", 128, 1.0)   # fp32 path: over 1.5 GB of scratch
    need = R.plan("chunkwise", w.torch_dtype, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk)[1]
    assert need > _lib.RET_NOALLOC_SCRATCH_BYTES
    q = torch.empty((w.B, w.H, w.L, w.d_k), dtype=torch.float32, device="cuda")
    v = torch.empty((w.B, w.H, w.L, w.d_v), dtype=torch.float32, device="cuda")
    inp = {"q": q, "k": q, "v": v, "state_in": None,
           "gamma": np.full(w.H, 0.99, np.float32), "theta": np.ones(w.d_k // 2, np.float32)}
    out = torch.empty_like(v)
    assert _noalloc(lib, inp, w, 0, out, None) == _lib.RET_EWORKSPACE
    assert R.sync_status() == R.RET_OK
