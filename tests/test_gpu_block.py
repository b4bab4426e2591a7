"""GPU parity of the MSR block around the core: the projection GEMM alone,
and the block (projections with the rotation folded into their epilogues,
the chunkwise core, GroupNorm with the swish gate, the output projection)
against the float64 oracle's msr_block on the same bf16 inputs."""

import numpy as np
import pytest
import torch

import linear_recurrent_sequence_prologue_b300 as R
from linear_recurrent_sequence_prologue_b300.inputs import gamma_schedule, theta_schedule, to_f64
from oracle import retention_ref as O

from helpers import assert_close, gpu_np, max_rel_inf

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrent_sequence_prologue_b300 import build
    build.build()
    R.load()


def _randn(gen, shape, std):
    return (torch.randn(*shape, generator=gen) * std).to(torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (300, 512, 192), (1000, 768, 320)])
def test_matmul_vs_float64(M, N, K):
    """C = A·W: fp32 output within fp32 accumulation error of the float64
    product of the same bf16 operands; bf16 output within the bf16 bound.
    M not a multiple of the 256-row tile checks the ragged rows."""
    gen = torch.Generator().manual_seed(M + N + K)
    a, w = _randn(gen, (M, K), 1.0), _randn(gen, (K, N), K ** -0.5)
    ref = to_f64(a) @ to_f64(w)
    c = R.matmul(a.cuda(), w.cuda(), out_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    assert max_rel_inf(gpu_np(c), ref) < 1e-5
    cb = R.matmul(a.cuda(), w.cuda())
    assert_close(gpu_np(cb), ref, torch.bfloat16, "matmul bf16")


def _block_inputs(B, L, D, H, d_k, d_v, D_out, seed):
    gen = torch.Generator().manual_seed(seed)
    x = _randn(gen, (B, L, D), 1.0)
    w = {"w_q": _randn(gen, (D, H, d_k), D ** -0.5), "w_k": _randn(gen, (D, H, d_k), D ** -0.5),
         "w_v": _randn(gen, (D, H, d_v), D ** -0.5), "w_g": _randn(gen, (D, H, d_v), D ** -0.5),
         "w_o": _randn(gen, (H, d_v, D_out), (H * d_v) ** -0.5)}
    s_in = torch.randn(B, H, d_k, d_v, generator=gen) * 0.1
    return x, w, s_in


@pytest.mark.parametrize("B,L,D,H,d_k,d_v,D_out,pos0", [
    (1, 300, 256, 2, 128, 256, 256, 5),     # ragged length, one-CTA core, 3 chunks
    (2, 256, 512, 2, 256, 512, 512, 0),     # CTA-pair core
    (1, 700, 256, 4, 64, 64, 256, 33),      # d_v = 64 (narrow value tile), 6 chunks
])
def test_msr_block_vs_oracle(B, L, D, H, d_k, d_v, D_out, pos0):
    x, w, s_in = _block_inputs(B, L, D, H, d_k, d_v, D_out, seed=L + D)
    gam, th = gamma_schedule(H), theta_schedule(d_k)
    dw = {k: v.cuda() for k, v in w.items()}
    z, s_out = R.msr_block(x.cuda(), dw["w_q"], dw["w_k"], dw["w_v"], dw["w_g"], dw["w_o"], gam, th,
                           pos0=pos0, state_in=s_in.cuda(), out_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    ref_z, ref_s = O.msr_block(to_f64(x), to_f64(w["w_q"]), to_f64(w["w_k"]), to_f64(w["w_v"]),
                               to_f64(w["w_g"]), to_f64(w["w_o"]), gam.astype(np.float64),
                               th.astype(np.float64), pos0, to_f64(s_in), 1e-5, 128)
    assert_close(gpu_np(z), ref_z, torch.bfloat16, "block z")
    assert_close(gpu_np(s_out), ref_s, torch.bfloat16, "block state")
    # The projections' epilogues write the chunk kernels' rotated operands:
    # the same bits as the front pass applied to bf16(x·W), so the final state
    # equals ret_chunkwise's on the projected q, k, v exactly.
    xf = x.cuda().reshape(B * L, D)
    heads = lambda t, d: t.reshape(B, L, H, d).permute(0, 2, 1, 3).contiguous()
    q = heads(R.matmul(xf, dw["w_q"].reshape(D, H * d_k)), d_k)
    k = heads(R.matmul(xf, dw["w_k"].reshape(D, H * d_k)), d_k)
    v = heads(R.matmul(xf, dw["w_v"].reshape(D, H * d_v)), d_v)
    _, s2 = R.chunkwise(q, k, v, gam, th, chunk=128, pos0=pos0, state_in=s_in.cuda())
    assert R.sync_status() == R.RET_OK
    assert torch.equal(s_out, s2)


def test_msr_block_state_chaining():
    """Two calls over the halves of a sequence, the state passed through and
    pos0 advanced, give the output of one call over the whole sequence (up
    to the bf16 rounding of the same operands)."""
    B, L, D, H, d_k, d_v, D_out = 1, 512, 256, 2, 128, 256, 256
    x, w, s_in = _block_inputs(B, L, D, H, d_k, d_v, D_out, seed=77)
    gam, th = gamma_schedule(H), theta_schedule(d_k)
    dw = {k: v.cuda() for k, v in w.items()}
    args = (dw["w_q"], dw["w_k"], dw["w_v"], dw["w_g"], dw["w_o"], gam, th)
    xc = x.cuda()
    z, s = R.msr_block(xc, *args, pos0=3, state_in=s_in.cuda(), out_dtype=torch.float32)
    za, sa = R.msr_block(xc[:, :256].contiguous(), *args, pos0=3, state_in=s_in.cuda(), out_dtype=torch.float32)
    zb, sb = R.msr_block(xc[:, 256:].contiguous(), *args, pos0=259, state_in=sa, out_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    assert torch.equal(torch.cat([za, zb], 1), z)
    assert torch.equal(sb, s)
