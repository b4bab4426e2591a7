"""The algorithmic work bench.py divides by: the figures the chunkwise form,
the decode step and the gradient pass fix for the workloads (no GPU)."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from linear_recurrent_sequence_prologue_b300.inputs import WORKLOADS  # noqa: E402


def test_chunkwise_work_at_the_7b_shape():
    w = WORKLOADS["msr7b"]
    # 2b·d_k + 2b·d_v + 4·d_k·d_v flop per token per head over B·H·L
    assert bench.chunk_flops(w) == 2 * 16 * 8192 * (2 * 128 * 256 + 2 * 128 * 512 + 4 * 256 * 512)
    assert abs(bench.chunk_flops(w) - 1.890e11) / 1.890e11 < 1e-3
    # q, k, v in and o out in bf16, state in and out in fp32
    assert bench.chunk_bytes(w) == 32 * 8192 * (2 * 256 + 2 * 512) * 2 + 2 * 32 * 256 * 512 * 4
    assert abs(bench.chunk_bytes(w) - 838.9e6) / 838.9e6 < 1e-3


def test_decode_bytes_per_step():
    w = WORKLOADS["decode"]
    assert abs(bench.decode_bytes(w) - 2.154e9) / 2.154e9 < 1e-3


def test_gradient_pass_work():
    w = WORKLOADS["msr7b"]
    f_out, f_ds = bench.backward_flops(w)
    assert f_out + f_ds == 3 * bench.chunk_flops(w)      # three evaluations of the form
    b = bench.backward_tc_bytes(w)
    n, L = 32, 8192
    # operand pass: q, k, v, dO read once; ω·dO and ζ·V (d_v wide), K̂′ and Q″
    # (d_k wide, folded), K′ and Q′ (d_k wide) written once each, all bf16
    reads = n * L * 2 * (2 * 256 + 2 * 512)
    writes = n * 2 * (2 * L * 512 + 2 * L * 256 + 2 * L * 256)
    assert b["bwd_prep"] == reads + writes
    # gradient outputs: two bf16 pieces of d_k in, bf16 dq and dk out (dv is
    # written by the chunk kernel)
    assert b["bwd_grad_out"] == n * L * 2 * (2 * 256 * 2 + 256 * 2)


def test_ffma_peak_from_unit_counts():
    # 148 SMs × 128 fp32 lanes × 2 flop per FFMA × 2.032 GHz, in TFLOP/s
    assert abs(bench.FFMA_TFLOPS - 148 * 128 * 2 * 2.032e-3) < 1e-9


def test_param_walk_bytes():
    # 7B shape: per walk the value rows (v or dO, bf16), the hi + lo operand
    # rows (4 bytes per element), 64 per-chunk fp32 states of 256 × 512 per
    # (b, h), and the state terms (S_in forward; S_in and dS_out backward)
    w = WORKLOADS["msr7b"]
    n, L, st = 32, 8192, 256 * 512 * 4
    rows, ops = n * L * 512 * 2, n * L * 256 * 4
    assert bench.param_walk_bytes(w) == (rows + ops + n * st + 64 * n * st) + (rows + ops + 64 * n * st + 2 * n * st)

