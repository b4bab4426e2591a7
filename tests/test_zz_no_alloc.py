"""ret_chunkwise_noalloc: the chunkwise entry point for callers that cannot
allocate device memory (plugins of a host that owns the device memory
budget, latency-critical loops).  It runs the same kernels as ret_chunkwise
with the library's built-in scratch array instead of a caller workspace.

Checked through the C ABI against ret_chunkwise, on two calls in a row with
different inputs (the shared array keeps the previous call's contents), on
both kernel paths, plus the size limit.  Collected last on purpose.
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


def _noalloc(lib, inp, w, pos0, out, state_out):
    g = np.ascontiguousarray(inp["gamma"], np.float32)
    t = np.ascontiguousarray(inp["theta"], np.float32)
    fp = lambda a: a.ctypes.data_as(C.POINTER(C.c_float))
    dt = _lib.RET_BF16 if inp["q"].dtype == torch.bfloat16 else _lib.RET_F32
    odt = _lib.RET_BF16 if out.dtype == torch.bfloat16 else _lib.RET_F32
    ptr = lambda x: None if x is None else C.c_void_p(x.data_ptr())
    st = lib.ret_chunkwise_noalloc(ptr(inp["q"]), ptr(inp["k"]), ptr(inp["v"]), dt, fp(g), fp(t),
                                   w.B, w.H, w.L, w.d_k, w.d_v, pos0, w.chunk,
                                   ptr(inp.get("state_in")), ptr(state_out), ptr(out), odt, None,
                                   C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


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
        inp = make_inputs(w, seed=seed)
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        ref_o, ref_s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"],
                                   chunk=w.chunk, pos0=3, state_in=d["state_in"])
        out = torch.full_like(ref_o, float("nan"))
        s_out = torch.full_like(ref_s, float("nan"))
        assert _noalloc(lib, d, w, 3, out, s_out) == _lib.RET_OK
        assert R.sync_status() == R.RET_OK
        assert_close(out.double().cpu().numpy(), ref_o.double().cpu().numpy(), w.torch_dtype, "out")
        assert_close(s_out.double().cpu().numpy(), ref_s.double().cpu().numpy(), w.torch_dtype, "state")


def test_noalloc_rejects_problems_beyond_the_array():
    lib = R.load()
    w = Workload("big", 2, 16, 8192, 256, 512, "bf16", 128, 1.0)   # needs 268 MB of scratch
    q = torch.empty((1,), dtype=torch.bfloat16, device="cuda")
    inp = {"q": q, "k": q, "v": q, "state_in": None,
           "gamma": np.full(w.H, 0.99, np.float32), "theta": np.ones(w.d_k // 2, np.float32)}
    out = torch.empty((1,), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, inp, w, 0, out, None) == _lib.RET_EWORKSPACE
