"""Shared helpers for the parity tests: tolerances and oracle slicing."""

import numpy as np
import torch

from linear_recurrent_sequence_prologue_b300.inputs import to_f64

# Tolerances of the contract: fp32 inputs → max|err| ≤ 1e-4·‖O‖∞;
# bf16 inputs with fp32 accumulation → relative Frobenius error ≤ 2e-2.
FP32_TOL = 1e-4
BF16_TOL = 2e-2
# Guards beside the whole-tensor bf16 bound, so that a few wrong rows or
# elements cannot hide inside a large tensor (one wrong row of 8192 moves the
# Frobenius error by only ~1/√8192):
# * every row (last axis: the d_v or d_k channels of one token, or one state
#   row) within the same relative error 2e-2 as the whole tensor; rows whose
#   reference norm is below 10% of the rows' RMS norm are measured against that
#   floor instead of their own norm.  Such a row is one whose few terms nearly
#   cancel (e.g. the first row of a gradient, one score times one vector, with
#   the score a dot product that happens to be small): the bf16 rounding of
#   the operands leaves an error of u times the size of the terms, not of
#   their cancelled sum, so its own relative error says nothing.  A missing
#   or garbage row of typical size is still off by ~1 against the floor;
# * every element within 2e-2·‖O‖∞.  The bf16 path rounds each operand once
#   (q″, k̂′, the masked scores, the carried state, the output; unit roundoff
#   u = 2^-8), so an element's error is a few u times the size of its terms;
#   at ‖O‖∞ ≈ 5× the RMS output that is ≈ 5e-3·‖O‖∞ at six standard deviations
#   over 10^8 elements (measured: ≈ 3e-3), and 2e-2 leaves a factor of four.
BF16_ROW_TOL = 2e-2
BF16_ELEM_TOL = 2e-2
ROW_FLOOR = 0.1


def gpu_np(t):
    return to_f64(t)


def max_rel_inf(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


def rel_fro(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def max_row_rel(got, ref):
    """Largest per-row relative error (rows = last axis), with the 10% floor."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if ref.ndim < 2:
        return rel_fro(got, ref)
    g = got.reshape(-1, ref.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(r, axis=1)
    rms = float(np.sqrt(np.mean(rn ** 2)))
    den = np.maximum(rn, max(ROW_FLOOR * rms, 1e-300))
    return float(np.max(np.linalg.norm(g - r, axis=1) / den))


def assert_close(got, ref, dtype, what=""):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} != {ref.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if dtype == torch.float32:
        e = max_rel_inf(got, ref)
        assert e <= FP32_TOL, f"{what}: max|err|/‖ref‖∞ = {e:.3e} > {FP32_TOL}"
    else:
        e = rel_fro(got, ref)
        assert e <= BF16_TOL, f"{what}: relative Frobenius error {e:.3e} > {BF16_TOL}"
        er = max_row_rel(got, ref)
        assert er <= BF16_ROW_TOL, f"{what}: worst row relative error {er:.3e} > {BF16_ROW_TOL}"
        ee = max_rel_inf(got, ref)
        assert ee <= BF16_ELEM_TOL, f"{what}: max|err|/‖ref‖∞ = {ee:.3e} > {BF16_ELEM_TOL}"
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
