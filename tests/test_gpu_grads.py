"""GPU parity of the training-side calls beside the gradient pass: the
gradients with respect to γ and θ (ret_chunkwise_param_grads, fed by the
library's own forward and backward calls) and the GroupNorm forward and
backward calls, against the float64 oracle on the same inputs."""

import numpy as np
import pytest
import torch

import linear_recurrent_sequence_prologue_b300 as R
from linear_recurrent_sequence_prologue_b300.inputs import Workload, make_grad_inputs, make_inputs, to_f64
from oracle import retention_ref as O

from helpers import BF16_TOL, FP32_TOL, assert_close, gpu_np, max_rel_inf, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrent_sequence_prologue_b300 import build
    build.build()
    R.load()


def _vec_close(got, ref, bf16, name):
    """One parameter-gradient vector: fp32 within 1e-4·max|ref| element-wise;
    bf16 operands within 2e-2 relative (Frobenius) and 2e-2·max|ref|
    element-wise (each entry is a sum over many tokens of products of
    once-rounded operands)."""
    if bf16:
        assert rel_fro(got, ref) <= BF16_TOL, (name, rel_fro(got, ref))
        assert max_rel_inf(got, ref) <= BF16_TOL, (name, max_rel_inf(got, ref))
    else:
        assert max_rel_inf(got, ref) <= FP32_TOL, (name, max_rel_inf(got, ref))


def _run_grads(w, pos0, chunk, out_dtype, grad_dtype, states, seed):
    inp = make_inputs(w, seed=seed)
    gi = make_grad_inputs(w, seed=seed + 1, d_state_std=1.0 if states else 0.0)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    s_in = inp["state_in"].cuda() if states else None
    d_out = gi["d_out"].cuda()
    d_so = gi["d_state_out"].cuda() if states else None
    out, s_out = R.chunkwise(q, k, v, inp["gamma"], inp["theta"], chunk=chunk, pos0=pos0, state_in=s_in,
                             out_dtype=out_dtype)
    dq, dk, dv, ds_in = R.chunkwise_backward(q, k, v, d_out, inp["gamma"], inp["theta"], chunk=chunk,
                                             pos0=pos0, state_in=s_in, d_state_out=d_so,
                                             grad_dtype=grad_dtype)
    dg, dt = R.param_grads(q, k, v, d_out, out, dq, dk, dv, inp["gamma"], inp["theta"], pos0=pos0,
                           state_in=s_in, d_state_out=d_so)
    assert R.sync_status() == R.RET_OK
    ref_g, ref_t = O.retention_param_grads(
        to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]), np.asarray(inp["gamma"], np.float64),
        np.asarray(inp["theta"], np.float64), pos0, to_f64(inp["state_in"]) if states else None,
        to_f64(gi["d_out"]), to_f64(gi["d_state_out"]) if states else None)
    return gpu_np(dg), gpu_np(dt), ref_g, ref_t


@pytest.mark.parametrize("dtype,B,H,L,d_k,d_v,chunk,pos0,states,out_dtype", [
    ("f32", 2, 3, 300, 32, 24, 32, 7, True, torch.float32),     # 16-byte rows, ragged chunks
    ("f32", 1, 2, 70, 6, 5, 16, 1000, True, torch.float32),     # element-by-element rows
    ("f32", 2, 2, 129, 16, 16, 64, 0, False, torch.float32),    # no state terms
    ("bf16", 1, 2, 384, 256, 256, 128, 5, True, torch.float32),     # tensor-core pair kernels
    ("bf16", 2, 2, 300, 128, 256, 128, 0, False, torch.bfloat16),   # bf16 out, ragged, one-CTA kernel
    ("bf16", 1, 2, 200, 48, 96, 32, 4, True, torch.float32),        # fp32 kernels, partial walk tiles
])
def test_param_grads_vs_oracle(dtype, B, H, L, d_k, d_v, chunk, pos0, states, out_dtype):
    w = Workload("custom", B, H, L, d_k, d_v, dtype, chunk, 1.0, state_std=0.1 if states else 0.0)
    gdt = torch.float32
    dg, dt, rg, rt = _run_grads(w, pos0, chunk, out_dtype, gdt, states, seed=L + d_k)
    bf16 = dtype == "bf16" or out_dtype == torch.bfloat16
    _vec_close(dg, rg, bf16, "d_gamma")
    _vec_close(dt, rt, bf16, "d_theta")


def test_param_grads_only_one_output_and_determinism():
    """Each output alone gives the same bits as both together, and two calls
    give the same bits (fixed-order sums)."""
    w = Workload("custom", 2, 2, 260, 64, 64, "f32", 64, 1.0, state_std=0.1)
    inp = make_inputs(w, seed=3)
    gi = make_grad_inputs(w, seed=4, d_state_std=1.0)
    q, k, v, s_in = (inp[n].cuda() for n in ("q", "k", "v", "state_in"))
    d_out, d_so = gi["d_out"].cuda(), gi["d_state_out"].cuda()
    out, s_out = R.chunkwise(q, k, v, inp["gamma"], inp["theta"], chunk=64, pos0=2, state_in=s_in)
    dq, dk, dv, ds_in = R.chunkwise_backward(q, k, v, d_out, inp["gamma"], inp["theta"], chunk=64, pos0=2,
                                             state_in=s_in, d_state_out=d_so)
    args = (q, k, v, d_out, out, dq, dk, dv, inp["gamma"], inp["theta"])
    kw = dict(pos0=2, state_in=s_in, d_state_out=d_so)
    g1, t1 = R.param_grads(*args, **kw)
    g2, t2 = R.param_grads(*args, **kw)
    g3, none_t = R.param_grads(*args, **kw, want_theta=False)
    none_g, t3 = R.param_grads(*args, **kw, want_gamma=False)
    assert R.sync_status() == R.RET_OK
    assert none_t is None and none_g is None
    assert torch.equal(g1, g2) and torch.equal(t1, t2)
    assert torch.equal(g1, g3) and torch.equal(t1, t3)


@pytest.mark.parametrize("L,states", [(300, True), (256, False), (1, True)])
def test_param_grads_tensor_core_walks_match_fp32_walks(L, states):
    """The tensor-core state walks (bf16 hi + lo operands, fp32 accumulation)
    against the fp32 walks on the same forward and gradient-pass outputs:
    ragged and whole chunks, one token, with and without state terms; two
    calls give the same bits."""
    w = Workload("custom", 2, 2, L, 256, 256, "bf16", 128, 1.0, state_std=0.1 if states else 0.0)
    inp = make_inputs(w, seed=7 + L)
    gi = make_grad_inputs(w, seed=8 + L, d_state_std=1.0 if states else 0.0)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    s_in = inp["state_in"].cuda() if states else None
    d_out = gi["d_out"].cuda()
    d_so = gi["d_state_out"].cuda() if states else None
    out, _ = R.chunkwise(q, k, v, inp["gamma"], inp["theta"], chunk=128, pos0=11, state_in=s_in,
                         out_dtype=torch.float32)
    dq, dk, dv, _ = R.chunkwise_backward(q, k, v, d_out, inp["gamma"], inp["theta"], chunk=128, pos0=11,
                                         state_in=s_in, d_state_out=d_so, grad_dtype=torch.float32)
    args = (q, k, v, d_out, out, dq, dk, dv, inp["gamma"], inp["theta"])
    kw = dict(pos0=11, state_in=s_in, d_state_out=d_so)
    g1, t1 = R.param_grads(*args, **kw)
    g2, t2 = R.param_grads(*args, **kw)
    R.force_path(R.RET_PATH_SIMT)
    try:
        gf, tf = R.param_grads(*args, **kw)
    finally:
        R.force_path(0)
    assert R.sync_status() == R.RET_OK
    assert torch.equal(g1, g2) and torch.equal(t1, t2)
    # 16 significant bits per walk operand against fp32: far inside the bf16 bound
    assert max_rel_inf(gpu_np(g1), gpu_np(gf)) <= 1e-3, (gpu_np(g1), gpu_np(gf))
    assert max_rel_inf(gpu_np(t1), gpu_np(tf)) <= 1e-3


@pytest.mark.parametrize("head", [0, 15])
def test_param_grads_7b_shape_full_length(head):
    """The 7B shape's batch (2 sequences of 8192 tokens, d_k 256, d_v 512,
    state_in and d_state_out) on one head at full length: the library's
    forward, gradient pass and parameter gradients against the oracle.  Head
    0 has the shortest decay window (γ = 1 − 2^-5), where summing with
    whole-sequence positions would amplify the bf16 rounding 256-fold; head
    15 the longest."""
    full = Workload("msr7b", 2, 16, 8192, 256, 512, "bf16", 128, 1.28, state_std=0.1)
    inp = make_inputs(full, seed=0)
    gi = make_grad_inputs(full, seed=1, d_state_std=1.0)
    sl = lambda t: t[:, head:head + 1].contiguous()
    q, k, v, s_in = (sl(inp[n]) for n in ("q", "k", "v", "state_in"))
    d_out, d_so = sl(gi["d_out"]), sl(gi["d_state_out"])
    gam = np.asarray(inp["gamma"][head:head + 1], np.float32)
    th = inp["theta"]
    qc, kc, vc, sc, dc, dsc = (t.cuda() for t in (q, k, v, s_in, d_out, d_so))
    out, _ = R.chunkwise(qc, kc, vc, gam, th, chunk=128, pos0=3, state_in=sc, out_dtype=torch.float32)
    dq, dk, dv, _ = R.chunkwise_backward(qc, kc, vc, dc, gam, th, chunk=128, pos0=3, state_in=sc,
                                         d_state_out=dsc, grad_dtype=torch.float32)
    dg, dt = R.param_grads(qc, kc, vc, dc, out, dq, dk, dv, gam, th, pos0=3, state_in=sc, d_state_out=dsc)
    assert R.sync_status() == R.RET_OK
    rg, rt = O.retention_param_grads(to_f64(q), to_f64(k), to_f64(v), gam.astype(np.float64),
                                     np.asarray(th, np.float64), 3, to_f64(s_in), to_f64(d_out),
                                     to_f64(d_so))
    assert abs(gpu_np(dg)[0] - rg[0]) <= BF16_TOL * abs(rg[0]), (gpu_np(dg), rg)
    _vec_close(gpu_np(dt), rt, True, "d_theta")


# ---------------------------------------------------------------- GroupNorm --
def _gn_inputs(B, H, L, d_v, dtype, seed, affine):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(B, H, L, d_v, generator=g) * 2 + 0.3).to(dtype)
    dy = torch.randn(B, H, L, d_v, generator=g).to(dtype)
    w = torch.randn(H, d_v, generator=g) if affine else None
    b = torch.randn(H, d_v, generator=g) if affine else None
    return x, dy, w, b


@pytest.mark.parametrize("B,H,L,d_v,dtype,affine", [
    (2, 3, 50, 48, torch.float32, True),
    (1, 2, 300, 512, torch.bfloat16, False),
    (1, 2, 33, 20, torch.float32, True),
    (1, 3, 47, 1024, torch.bfloat16, True),     # 32 channels a lane, one row per warp at a time
    (3, 1, 23, 256, torch.bfloat16, True),      # rows not a multiple of the rows a warp takes
    (1, 2, 41, 512, torch.float32, True),       # fp32 rows: two 16-byte vectors per 8 channels
])
def test_groupnorm_call_vs_oracle(B, H, L, d_v, dtype, affine):
    x, _, w, b = _gn_inputs(B, H, L, d_v, dtype, 5 + d_v, affine)
    dw = w.cuda() if affine else None
    db = b.cuda() if affine else None
    y = R.groupnorm(x.cuda(), 1e-5, dw, db, out_dtype=torch.float32)
    ref = O.group_norm(to_f64(x), 1e-5, to_f64(w) if affine else None, to_f64(b) if affine else None)
    assert R.sync_status() == R.RET_OK
    assert_close(gpu_np(y), ref, torch.float32, "groupnorm")
    xc = x.cuda()
    y2 = R.groupnorm(xc, 1e-5, dw, db, out=xc)   # in place
    assert R.sync_status() == R.RET_OK
    assert_close(gpu_np(y2), ref, dtype, "groupnorm in place")


@pytest.mark.parametrize("B,H,L,d_v,dtype,gdtype,affine", [
    (2, 3, 70, 48, torch.float32, torch.float32, True),        # 16-byte rows, 8 per lane
    (1, 2, 90, 20, torch.float32, torch.float32, True),        # element by element
    (2, 2, 200, 512, torch.bfloat16, torch.float32, True),     # 16 per lane
    (1, 2, 65, 1024, torch.float32, torch.bfloat16, False),    # 32 per lane, bf16 gradient
    (1, 1, 40, 100, torch.bfloat16, torch.bfloat16, False),    # ragged width
])
def test_groupnorm_backward_vs_oracle(B, H, L, d_v, dtype, gdtype, affine):
    x, dy, w, _ = _gn_inputs(B, H, L, d_v, dtype, 11 + d_v, affine)
    d_x, d_w, d_b = R.groupnorm_backward(x.cuda(), dy.cuda(), 1e-5, w.cuda() if affine else None,
                                         grad_dtype=gdtype)
    assert R.sync_status() == R.RET_OK
    r_x, r_w, r_b = O.groupnorm_backward(to_f64(x), to_f64(dy), 1e-5, to_f64(w) if affine else None)
    tol = torch.float32 if gdtype == torch.float32 else torch.bfloat16
    assert_close(gpu_np(d_x), r_x, tol, "d_x")
    for got, ref, name in ((d_w, r_w, "d_weight"), (d_b, r_b, "d_bias")):
        assert max_rel_inf(gpu_np(got), ref) <= FP32_TOL, name


def test_groupnorm_backward_1p3b_shape():
    """The 1.3B shape (8·8·2048 rows of 512 channels, bf16) against the
    oracle on every row and channel."""
    x, dy, w, _ = _gn_inputs(8, 8, 2048, 512, torch.bfloat16, 77, True)
    d_x, d_w, d_b = R.groupnorm_backward(x.cuda(), dy.cuda(), 1e-5, w.cuda(), grad_dtype=torch.bfloat16)
    assert R.sync_status() == R.RET_OK
    r_x, r_w, r_b = O.groupnorm_backward(to_f64(x), to_f64(dy), 1e-5, to_f64(w))
    assert_close(gpu_np(d_x), r_x, torch.bfloat16, "d_x")
    assert max_rel_inf(gpu_np(d_w), r_w) <= FP32_TOL
    assert max_rel_inf(gpu_np(d_b), r_b) <= FP32_TOL


def test_training_chain_with_groupnorm():
    """Forward without GroupNorm + ret_groupnorm, then ret_groupnorm_backward
    + the gradient pass + the parameter gradients: the composition against
    the oracle's chain (GroupNorm backward feeding retention_backward)."""
    w = Workload("custom", 1, 2, 200, 64, 64, "f32", 32, 1.0, state_std=0.1)
    inp = make_inputs(w, seed=8)
    g = torch.Generator().manual_seed(9)
    dz = torch.randn(1, 2, 200, 64, generator=g)
    gw = torch.randn(2, 64, generator=g)
    q, k, v, s_in = (inp[n].cuda() for n in ("q", "k", "v", "state_in"))
    o, _ = R.chunkwise(q, k, v, inp["gamma"], inp["theta"], chunk=32, pos0=4, state_in=s_in)
    z = R.groupnorm(o, 1e-5, gw.cuda())
    d_o, d_w, _ = R.groupnorm_backward(o, dz.cuda(), 1e-5, gw.cuda())
    dq, dk, dv, ds_in = R.chunkwise_backward(q, k, v, d_o, inp["gamma"], inp["theta"], chunk=32, pos0=4,
                                             state_in=s_in)
    dg, dt = R.param_grads(q, k, v, d_o, o, dq, dk, dv, inp["gamma"], inp["theta"], pos0=4, state_in=s_in)
    assert R.sync_status() == R.RET_OK
    args = [to_f64(inp[n]) for n in ("q", "k", "v")]
    gam, th = np.asarray(inp["gamma"], np.float64), np.asarray(inp["theta"], np.float64)
    ro, _ = O.retention(*args, gam, th, 4, to_f64(inp["state_in"]), "chunkwise", 32)
    rz = O.group_norm(ro, 1e-5, to_f64(gw))
    rdo, rdw, _ = O.groupnorm_backward(ro, to_f64(dz), 1e-5, to_f64(gw))
    rdq, rdk, rdv, rds = O.retention_backward(*args, gam, th, 4, to_f64(inp["state_in"]), rdo)
    rg, rt = O.retention_param_grads(*args, gam, th, 4, to_f64(inp["state_in"]), rdo)
    assert_close(gpu_np(z), rz, torch.float32, "z")
    assert max_rel_inf(gpu_np(d_w), rdw) <= FP32_TOL
    for got, ref, name in ((dq, rdq, "dq"), (dk, rdk, "dk"), (dv, rdv, "dv"), (ds_in, rds, "dS_in")):
        assert_close(gpu_np(got), ref, torch.float32, name)
    _vec_close(gpu_np(dg), rg, False, "d_gamma")
    _vec_close(gpu_np(dt), rt, False, "d_theta")
