"""Shared helpers for the parity tests: tolerances and oracle slicing."""

import numpy as np
import torch

from linear_recurrent_sequence_prologue_b300.inputs import to_f64

# Tolerances of the contract: fp32 inputs → max|err| ≤ 1e-4·‖O‖∞;
# bf16 inputs with fp32 accumulation → relative Frobenius error ≤ 2e-2.
FP32_TOL = 1e-4
BF16_TOL = 2e-2


def gpu_np(t):
    return to_f64(t)


def max_rel_inf(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


def rel_fro(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def assert_close(got, ref, dtype, what=""):
    if dtype == torch.float32:
        e = max_rel_inf(got, ref)
        assert e <= FP32_TOL, f"{what}: max|err|/‖ref‖∞ = {e:.3e} > {FP32_TOL}"
    else:
        e = rel_fro(got, ref)
        assert e <= BF16_TOL, f"{what}: relative Frobenius error {e:.3e} > {BF16_TOL}"
    return e


def head_slice(inp, b, h):
    """Inputs of one (b, h) pair, as float64 arrays shaped for the oracle."""
    q = to_f64(inp["q"][b:b + 1, h:h + 1])
    k = to_f64(inp["k"][b:b + 1, h:h + 1])
    v = to_f64(inp["v"][b:b + 1, h:h + 1])
    s = None if inp.get("state_in") is None else to_f64(inp["state_in"][b:b + 1, h:h + 1])
    g = np.asarray(inp["gamma"], np.float64)[h:h + 1]
    th = np.asarray(inp["theta"], np.float64)
    return q, k, v, s, g, th
