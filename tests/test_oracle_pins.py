"""Pins of the float64 oracle against things other than itself.

Each check ties the oracle to a passage of the RetNet pages, a closed form, a
library routine or a brute-force evaluation; ``test_mutants_are_caught``
plants plausible mistakes in the oracle's source and checks that at least
one pin fails for every one of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import retention_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed=0, B=2, H=2, L=7, d_k=4, d_v=3, state=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, L, d_k))
    k = rng.standard_normal((B, H, L, d_k))
    v = rng.standard_normal((B, H, L, d_v))
    gamma = rng.uniform(0.3, 0.95, size=H)
    theta = rng.uniform(0.1, 2.0, size=d_k // 2)
    S = rng.standard_normal((B, H, d_k, d_v)) if state else None
    return q, k, v, gamma, theta, S


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b))))


# ----------------------------------------------------------------------------
# Pins, written as functions so that the mutation test can rerun them.
# Each returns None on success and raises AssertionError on failure.
# ----------------------------------------------------------------------------

def pin_demo_parallel_equals_recurrent():
    """RetNet 保留网络 explainer, 'Python 演示': parallel ≡ recurrent, err < 1e-8."""
    cfg = json.load(open(os.path.join(GOLDEN, "demo_parallel_recurrent.json")))
    rs = np.random.RandomState(cfg["seed"])
    n, dim, g = cfg["n"], cfg["dim"], cfg["gamma"]
    x = rs.randn(n, dim)
    wq, wk, wv = rs.randn(dim, dim), rs.randn(dim, dim), rs.randn(dim, dim)
    q, k, v = (x @ w for w in (wq, wk, wv))
    op, _ = R.parallel_core(q[None, None], k[None, None], v[None, None], [g])
    orr, _ = R.recurrent_core(q[None, None], k[None, None], v[None, None], [g])
    assert np.abs(op - orr).max() < cfg["max_abs_err"]


def pin_rotation_fixed_angles():
    """«从RoPE到Retention…» §2 theta_shift at angles k·π/2, worked by hand."""
    cases = json.load(open(os.path.join(GOLDEN, "rotation_cases.json")))["cases"]
    for c in cases:
        x = np.array(c["x"])[None, :]
        sin, cos = R.rotation_tables([c["n"]], c["theta"])
        y = R.theta_shift(x, sin, cos)[0]
        assert np.allclose(y, c["expect"], atol=1e-12), (c, y)


def pin_retention_hand_case():
    """A two-token case worked by hand from the definitions (golden file)."""
    c = json.load(open(os.path.join(GOLDEN, "rotation_cases.json")))["retention_cases"][0]
    q = np.array(c["q"])[None, None]
    k = np.array(c["k"])[None, None]
    v = np.array(c["v"])[None, None]
    for form, chunk in (("parallel", None), ("recurrent", None), ("chunkwise", 1), ("chunkwise", 2)):
        o, S = R.retention(q, k, v, [c["gamma"]], c["theta"], c["pos0"], None, form, chunk)
        assert np.allclose(o[0, 0], c["out"], atol=1e-12), (form, o)
        assert np.allclose(S[0, 0], c["state"], atol=1e-12), (form, S)
    o, S = R.brute_force(q, k, v, [c["gamma"]], c["theta"], c["pos0"])
    assert np.allclose(o[0, 0], c["out"], atol=1e-12)
    assert np.allclose(S[0, 0], c["state"], atol=1e-12)


def pin_forms_match_brute_force():
    """Parallel, recurrent and chunkwise (several b) equal the scalar double loop."""
    for seed, pos0, state in ((0, 0, False), (1, 5, True), (2, 123, True)):
        q, k, v, g, th, S = _rand_case(seed, state=state)
        ob, Sb = R.brute_force(q, k, v, g, th, pos0, S)
        for form, chunk in (("parallel", None), ("recurrent", None), ("chunkwise", 1),
                            ("chunkwise", 2), ("chunkwise", 3), ("chunkwise", 7)):
            o, Sx = R.retention(q, k, v, g, th, pos0, S, form, chunk)
            assert _rel(o, ob) < 1e-12, (form, chunk, _rel(o, ob))
            assert _rel(Sx, Sb) < 1e-12, (form, chunk, _rel(Sx, Sb))


def pin_linear_attention_limit():
    """γ = 1, θ = 0: causal linear attention, o_t = q_t·Σ_{m≤t} k_mᵀv_m/√d + q_t S_in (cumsum)."""
    q, k, v, _, th, S = _rand_case(3, L=9)
    H, d_k = q.shape[1], q.shape[-1]
    kv = np.einsum("bhtk,bhtv->bhtkv", k, v) / math.sqrt(d_k)
    cum = np.cumsum(kv, axis=2) + S[:, :, None]
    expect = np.einsum("bhtk,bhtkv->bhtv", q, cum)
    for form, chunk in (("parallel", None), ("recurrent", None), ("chunkwise", 4)):
        o, Sx = R.retention(q, k, v, np.ones(H), np.zeros_like(th), 0, S, form, chunk)
        assert _rel(o, expect) < 1e-12
        assert _rel(Sx, cum[:, :, -1]) < 1e-12
    o, _ = R.brute_force(q, k, v, np.ones(H), np.zeros_like(th), 0, S)
    assert _rel(o, expect) < 1e-12


def pin_gamma_zero():
    """γ = 0: only the diagonal survives (0⁰ = 1): o_t = (q′_t·k′_t) v_t; S_out = k′_{L−1}ᵀ v_{L−1}."""
    q, k, v, _, th, S = _rand_case(4, L=6)
    H = q.shape[1]
    qp, kp = R.prologue(q, k, th, 7)
    expect = np.einsum("bhtk,bhtk->bht", qp, kp)[..., None] * v
    exS = kp[:, :, -1, :, None] * v[:, :, -1, None, :]
    for form, chunk in (("parallel", None), ("recurrent", None), ("chunkwise", 4)):
        o, Sx = R.retention(q, k, v, np.zeros(H), th, 7, S, form, chunk)
        assert _rel(o, expect) < 1e-12
        assert _rel(Sx, exS) < 1e-12
    o, Sb = R.brute_force(q, k, v, np.zeros(H), th, 7, S)
    assert _rel(o, expect) < 1e-12 and _rel(Sb, exS) < 1e-12


def pin_single_token():
    """L = 1: o = (q′·k′)v + γ q′ S_in; S_out = γ S_in + k′ᵀv."""
    q, k, v, g, th, S = _rand_case(5, L=1)
    qp, kp = R.prologue(q, k, th, 11)
    ex = (np.einsum("bhtk,bhtk->bht", qp, kp)[..., None] * v
          + g[None, :, None, None] * np.einsum("bhtk,bhkv->bhtv", qp, S))
    exS = g[None, :, None, None] * S + kp[:, :, 0, :, None] * v[:, :, 0, None, :]
    for form in ("parallel", "recurrent", "chunkwise"):
        o, Sx = R.retention(q, k, v, g, th, 11, S, form, 1)
        assert _rel(o, ex) < 1e-12 and _rel(Sx, exS) < 1e-12


def pin_theta_zero_is_identity():
    q, k, *_ = _rand_case(6)
    qp, kp = R.prologue(q, k, np.zeros(q.shape[-1] // 2), 99)
    assert np.array_equal(qp, q)
    assert np.allclose(kp, k / math.sqrt(q.shape[-1]), rtol=0, atol=1e-15)


def pin_rotation_preserves_pair_norms():
    q, _, _, _, th, _ = _rand_case(7)
    sin, cos = R.rotation_tables(np.arange(q.shape[2]) + 1000, th)
    y = R.theta_shift(q, sin, cos)
    n0 = q[..., 0::2] ** 2 + q[..., 1::2] ** 2
    n1 = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.allclose(n0, n1, rtol=1e-12, atol=0)


def pin_position_shift_invariance():
    """Only n − m matters (Θ on Q, Θ̄ on K ⇒ relative position): pos0 does not change O."""
    q, k, v, g, th, _ = _rand_case(8)
    o0, S0 = R.retention(q, k, v, g, th, 0, None, "chunkwise", 3)
    o1, _ = R.retention(q, k, v, g, th, 41, None, "chunkwise", 3)
    assert _rel(o1, o0) < 1e-11
    ob, _ = R.brute_force(q, k, v, g, th, 41)
    assert _rel(ob, o0) < 1e-11


def pin_exact_causality():
    """D_nm = 0 for n < m: outputs before m are bit-identical when later inputs change."""
    q, k, v, g, th, S = _rand_case(9, L=12)
    m = 5
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    rng = np.random.default_rng(99)
    q2[:, :, m:] = rng.standard_normal(q2[:, :, m:].shape) * 100
    k2[:, :, m:] = rng.standard_normal(k2[:, :, m:].shape) * 100
    v2[:, :, m:] = rng.standard_normal(v2[:, :, m:].shape) * 100
    for form, chunk in (("parallel", None), ("recurrent", None), ("chunkwise", 4), ("chunkwise", 5)):
        o1, _ = R.retention(q, k, v, g, th, 3, S, form, chunk)
        o2, _ = R.retention(q2, k2, v2, g, th, 3, S, form, chunk)
        assert np.array_equal(o1[:, :, :m], o2[:, :, :m]), form
        assert not np.array_equal(o1[:, :, m:], o2[:, :, m:])


def pin_chunk_limits():
    """b = 1 reduces to the recurrent form and b = L to the parallel form (分块循环)."""
    q, k, v, g, th, S = _rand_case(10, L=10)
    orec, Srec = R.retention(q, k, v, g, th, 2, S, "recurrent")
    opar, Spar = R.retention(q, k, v, g, th, 2, S, "parallel")
    o1, S1 = R.retention(q, k, v, g, th, 2, S, "chunkwise", 1)
    oL, SL = R.retention(q, k, v, g, th, 2, S, "chunkwise", 10)
    assert _rel(o1, orec) < 1e-12 and _rel(S1, Srec) < 1e-12
    assert _rel(oL, opar) < 1e-12 and _rel(SL, Spar) < 1e-12


def pin_split_call():
    """One call over [0, L) equals two calls over halves with the state passed through."""
    q, k, v, g, th, S = _rand_case(11, L=12)
    o, Sx = R.retention(q, k, v, g, th, 4, S, "chunkwise", 3)
    h = 6
    oa, Sa = R.retention(q[:, :, :h], k[:, :, :h], v[:, :, :h], g, th, 4, S, "chunkwise", 3)
    ob, Sb = R.retention(q[:, :, h:], k[:, :, h:], v[:, :, h:], g, th, 4 + h, Sa, "chunkwise", 3)
    assert _rel(np.concatenate([oa, ob], axis=2), o) < 1e-12
    assert _rel(Sb, Sx) < 1e-12


def pin_ragged_tail():
    q, k, v, g, th, S = _rand_case(12, L=11)
    opar, Spar = R.retention(q, k, v, g, th, 0, S, "parallel")
    for chunk in (2, 3, 4, 5, 6, 10):
        o, Sx = R.retention(q, k, v, g, th, 0, S, "chunkwise", chunk)
        assert _rel(o, opar) < 1e-12 and _rel(Sx, Spar) < 1e-12


def pin_linearity():
    q, k, v, g, th, S = _rand_case(13)
    v2 = np.random.default_rng(1).standard_normal(v.shape)
    S2 = np.random.default_rng(2).standard_normal(S.shape)
    oa, Sa = R.retention(q, k, v, g, th, 0, S, "chunkwise", 3)
    ob, Sb = R.retention(q, k, v2, g, th, 0, S2, "chunkwise", 3)
    oc, Sc = R.retention(q, k, 2.0 * v - 3.0 * v2, g, th, 0, 2.0 * S - 3.0 * S2, "chunkwise", 3)
    assert _rel(oc, 2.0 * oa - 3.0 * ob) < 1e-12
    assert _rel(Sc, 2.0 * Sa - 3.0 * Sb) < 1e-12


def pin_decode_steps_equal_recurrent():
    q, k, v, g, th, S = _rand_case(14, L=8)
    orec, Srec = R.retention(q, k, v, g, th, 20, S, "recurrent")
    st = S.copy()
    for t in range(q.shape[2]):
        o, st = R.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], g, th, 20 + t, st)
        assert _rel(o, orec[:, :, t]) < 1e-12
    assert _rel(st, Srec) < 1e-12


def pin_groupnorm_matches_torch():
    """Per-head GroupNorm equals torch.nn.functional.group_norm (float64, CPU)."""
    rng = np.random.default_rng(15)
    B, H, L, d_v = 2, 3, 5, 8
    o = rng.standard_normal((B, H, L, d_v)) * 3 + 1
    w = rng.standard_normal((H, d_v))
    b = rng.standard_normal((H, d_v))
    y = R.group_norm(o, 1e-5, w, b)
    x = torch.from_numpy(o).permute(0, 2, 1, 3).reshape(B * L, H * d_v)
    t = torch.nn.functional.group_norm(x, H, torch.from_numpy(w.reshape(-1)),
                                       torch.from_numpy(b.reshape(-1)), eps=1e-5)
    t = t.reshape(B, L, H, d_v).permute(0, 2, 1, 3).numpy()
    assert _rel(y, t) < 1e-12
    y0 = R.group_norm(o, 1e-5)
    assert np.allclose(y0.mean(-1), 0, atol=1e-12)
    assert np.allclose(y0.var(-1), 1, atol=1e-4)


def _backward_fd_check(with_state, with_dso, pos0):
    """retention_backward against central differences of the forward oracle,
    for the scalar <dO, out> + <dS_out, S_out>: every gradient term
    (intra-chunk scores, the state_in term, the state_out path, the rotation
    adjoint and the 1/√d_k scale) enters one of the four checks."""
    rng = np.random.default_rng(7 + pos0)
    B, H, L, d_k, d_v = 1, 2, 6, 4, 3
    q, k = rng.standard_normal((B, H, L, d_k)), rng.standard_normal((B, H, L, d_k))
    v = rng.standard_normal((B, H, L, d_v))
    S0 = 0.3 * rng.standard_normal((B, H, d_k, d_v)) if with_state else None
    g, th = np.array([0.9, 0.6]), np.array([0.4, 1.3])
    dO = rng.standard_normal((B, H, L, d_v))
    dSo = rng.standard_normal((B, H, d_k, d_v)) if with_dso else None

    def f(q_, k_, v_, s_):
        o, S = R.retention(q_, k_, v_, g, th, pos0, s_, "parallel")
        return (o * dO).sum() + ((S * dSo).sum() if with_dso else 0.0)

    grads = R.retention_backward(q, k, v, g, th, pos0, S0, dO, dSo)
    args = [q, k, v, S0 if with_state else np.zeros((B, H, d_k, d_v))]
    eps = 1e-6
    for which in range(4 if with_state else 3):
        x = args[which]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            a = [t.copy() for t in args]
            a[which][idx] += eps
            fp = f(*(a[:3] + [a[3] if with_state else None]))
            a[which][idx] -= 2 * eps
            fm = f(*(a[:3] + [a[3] if with_state else None]))
            num[idx] = (fp - fm) / (2 * eps)
        assert np.max(np.abs(num - grads[which])) < 1e-6, which
    if not with_state:   # d_state_in is still defined: the gradient at S_in = 0
        num = np.zeros((B, H, d_k, d_v))
        for idx in np.ndindex(num.shape):
            e = np.zeros_like(num)
            e[idx] = eps
            num[idx] = (f(q, k, v, e) - f(q, k, v, -e)) / (2 * eps)
        assert np.max(np.abs(num - grads[3])) < 1e-6


def pin_backward_finite_differences():
    _backward_fd_check(True, True, 11)
    _backward_fd_check(False, False, 0)


def _param_grads_fd_check(with_states, pos0):
    """retention_param_grads against central differences in γ and θ of the
    scalar <dO, out> + <dS_out, S_out>, the forward taken in the chunkwise
    form with a ragged last chunk (B = 2: the gradients sum over the batch)."""
    rng = np.random.default_rng(19 + pos0)
    B, H, L, d_k, d_v = 2, 2, 7, 4, 3
    q, k = rng.standard_normal((B, H, L, d_k)), rng.standard_normal((B, H, L, d_k))
    v = rng.standard_normal((B, H, L, d_v))
    S0 = 0.3 * rng.standard_normal((B, H, d_k, d_v)) if with_states else None
    dO = rng.standard_normal((B, H, L, d_v))
    dSo = rng.standard_normal((B, H, d_k, d_v)) if with_states else None
    g, th = np.array([0.9, 0.6]), np.array([0.4, 1.3])

    def f(g_, th_):
        o, S = R.retention(q, k, v, g_, th_, pos0, S0, "chunkwise", 3)
        return (o * dO).sum() + ((S * dSo).sum() if with_states else 0.0)

    dg, dth = R.retention_param_grads(q, k, v, g, th, pos0, S0, dO, dSo)
    eps = 1e-6
    for i in range(2):
        e = eps * np.eye(2)[i]
        num_g = (f(g + e, th) - f(g - e, th)) / (2 * eps)
        num_t = (f(g, th + e) - f(g, th - e)) / (2 * eps)
        assert abs(num_g - dg[i]) < 1e-6 * max(1.0, abs(num_g)), ("gamma", i)
        assert abs(num_t - dth[i]) < 1e-6 * max(1.0, abs(num_t)), ("theta", i)


def pin_param_grads_finite_differences():
    _param_grads_fd_check(True, 5)
    _param_grads_fd_check(False, 0)


def pin_theta_grad_position_shift_invariance():
    """Without state terms the output depends on θ only through (n − m)·θ,
    so the θ gradient is the same at every start position."""
    rng = np.random.default_rng(23)
    B, H, L, d_k, d_v = 1, 2, 9, 6, 2
    q, k = rng.standard_normal((B, H, L, d_k)), rng.standard_normal((B, H, L, d_k))
    v, dO = rng.standard_normal((B, H, L, d_v)), rng.standard_normal((B, H, L, d_v))
    g, th = np.array([0.8, 0.97]), np.array([0.3, 0.05, 1.1])
    _, a = R.retention_param_grads(q, k, v, g, th, 0, None, dO, None)
    _, b = R.retention_param_grads(q, k, v, g, th, 1000, None, dO, None)
    assert np.max(np.abs(a - b)) < 1e-9 * np.max(np.abs(a))
    assert np.max(np.abs(a)) > 1e-3


def pin_gamma_grad_single_token():
    """One token: out = (q′·k′)v + γ·q′S_in, S_out = γS_in + k′ᵀv.  So with
    no state the γ gradient is exactly 0, and with state_in and dS_out it
    is Σ dO·(q′S_in) + <dS_out, S_in>."""
    rng = np.random.default_rng(29)
    q, k = rng.standard_normal((2, 1, 1, 4)), rng.standard_normal((2, 1, 1, 4))
    v, dO = rng.standard_normal((2, 1, 1, 3)), rng.standard_normal((2, 1, 1, 3))
    S0, dSo = rng.standard_normal((2, 1, 4, 3)), rng.standard_normal((2, 1, 4, 3))
    g, th = np.array([0.7]), np.array([0.5, 2.0])
    dg0, _ = R.retention_param_grads(q, k, v, g, th, 3, None, dO, None)
    assert dg0[0] == 0.0
    dg, _ = R.retention_param_grads(q, k, v, g, th, 3, S0, dO, dSo)
    qp, _ = R.prologue(q, k, th, 3)
    ref = np.sum(dO[:, 0, 0] * np.einsum("bk,bkv->bv", qp[:, 0, 0], S0[:, 0])) + np.sum(dSo * S0)
    assert abs(dg[0] - ref) < 1e-12 * max(1.0, abs(ref))


def pin_groupnorm_backward():
    """groupnorm_backward against central differences of <d_y, group_norm(o)>
    in o, weight and bias, and against torch autograd of
    torch.nn.functional.group_norm (float64, one group per head)."""
    rng = np.random.default_rng(31)
    B, H, L, d_v = 2, 2, 3, 5
    o = rng.standard_normal((B, H, L, d_v)) * 2 + 0.5
    w, b = rng.standard_normal((H, d_v)), rng.standard_normal((H, d_v))
    dy = rng.standard_normal((B, H, L, d_v))
    d_o, d_w, d_b = R.groupnorm_backward(o, dy, 1e-3, w)
    f = lambda o_, w_, b_: np.sum(dy * R.group_norm(o_, 1e-3, w_, b_))
    eps = 1e-6
    for x, ref, which in ((o, d_o, 0), (w, d_w, 1), (b, d_b, 2)):
        for idx in np.ndindex(x.shape):
            a = [o.copy(), w.copy(), b.copy()]
            a[which][idx] += eps
            fp = f(*a)
            a[which][idx] -= 2 * eps
            num = (fp - f(*a)) / (2 * eps)
            assert abs(num - ref[idx]) < 1e-6 * max(1.0, abs(num)), (which, idx)
    x = torch.from_numpy(o).permute(0, 2, 1, 3).reshape(B * L, H * d_v).requires_grad_(True)
    tw = torch.from_numpy(w.reshape(-1)).requires_grad_(True)
    tb = torch.from_numpy(b.reshape(-1)).requires_grad_(True)
    y = torch.nn.functional.group_norm(x, H, tw, tb, eps=1e-3)
    y.backward(torch.from_numpy(dy).permute(0, 2, 1, 3).reshape(B * L, H * d_v))
    t_do = x.grad.reshape(B, L, H, d_v).permute(0, 2, 1, 3).numpy()
    assert _rel(d_o, t_do) < 1e-12
    assert _rel(d_w, tw.grad.reshape(H, d_v).numpy()) < 1e-12
    assert _rel(d_b, tb.grad.reshape(H, d_v).numpy()) < 1e-12


# Row-normalised decay (R9)
def pin_decay_row_sums_geometric_series():
    """r_N = Σ_{i≤N} γ^i is the geometric series (1 − γ^{N+1}) / (1 − γ); N + 1 at γ = 1."""
    g = np.array([0.9, 0.999, 1.0])
    r = R.decay_row_sums(g, 5, 40)
    N = np.arange(5, 45)
    for h, gh in enumerate(g):
        ref = N + 1.0 if gh == 1.0 else (1 - gh ** (N + 1)) / (1 - gh)
        assert np.allclose(r[h], ref, rtol=1e-13, atol=0)


def pin_normalised_gamma_one_is_a_running_mean():
    """γ = 1, θ = 0: o_t = q_t · (Σ_{m≤t} k′_mᵀ v_m) / (t + 1), a cumulative mean."""
    rng = np.random.default_rng(31)
    q, k, v = rng.standard_normal((1, 1, 12, 4)), rng.standard_normal((1, 1, 12, 4)), rng.standard_normal((1, 1, 12, 3))
    out = R.normalised_retention(q, k, v, np.array([1.0]), np.zeros(2))
    kv = np.cumsum(np.einsum("td,te->tde", k[0, 0] / 2.0, v[0, 0]), axis=0)   # k′ = k/√4
    ref = np.einsum("td,tde->te", q[0, 0], kv) / np.arange(1, 13)[:, None]
    assert np.allclose(out[0, 0], ref, rtol=1e-12, atol=1e-12)


def pin_normalised_cancels_under_groupnorm():
    """GroupNorm is invariant to a positive per-(token, head) scale ([P5]): with
    eps = 0 the normalised and the plain outputs agree after it; without it
    they differ by exactly r_t per row."""
    rng = np.random.default_rng(32)
    q, k = rng.standard_normal((2, 2, 20, 8)), rng.standard_normal((2, 2, 20, 8))
    v, s = rng.standard_normal((2, 2, 20, 6)), 0.1 * rng.standard_normal((2, 2, 8, 6))
    g, th = np.array([0.95, 0.7]), rng.uniform(0.01, 1, 4)
    a = R.normalised_retention(q, k, v, g, th, 3, s, gn={"eps": 0.0})
    b, _ = R.retention(q, k, v, g, th, 3, s, "parallel", gn={"eps": 0.0})
    assert np.allclose(a, b, rtol=1e-10, atol=1e-10)
    a = R.normalised_retention(q, k, v, g, th, 3, s)
    b, _ = R.retention(q, k, v, g, th, 3, s, "parallel")
    N = np.arange(3, 23)
    r = (1 - g[:, None] ** (N + 1)) / (1 - g[:, None])          # geometric series
    assert np.allclose(a * r[None, :, :, None], b, rtol=1e-12, atol=1e-12)


def pin_normalised_split_calls():
    """Positions are absolute: [0, L) in one call equals [0, L/2) then [L/2, L)
    with the state passed through and pos0 = L/2."""
    rng = np.random.default_rng(33)
    q, k, v = rng.standard_normal((1, 2, 24, 4)), rng.standard_normal((1, 2, 24, 4)), rng.standard_normal((1, 2, 24, 5))
    g, th = np.array([0.9, 0.99]), rng.uniform(0.01, 1, 2)
    whole = R.normalised_retention(q, k, v, g, th)
    first = R.normalised_retention(q[:, :, :12], k[:, :, :12], v[:, :, :12], g, th)
    _, S = R.retention(q[:, :, :12], k[:, :, :12], v[:, :, :12], g, th, 0, None, "parallel")
    second = R.normalised_retention(q[:, :, 12:], k[:, :, 12:], v[:, :, 12:], g, th, 12, S)
    assert np.allclose(whole, np.concatenate([first, second], axis=2), rtol=1e-12, atol=1e-12)


# MSR block around the core (R10)
def _block_inputs(seed, B=2, L=10, D=12, H=3, d_k=4, d_v=5, D_out=7):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((B, L, D)), w_q=rng.standard_normal((D, H, d_k)),
                w_k=rng.standard_normal((D, H, d_k)), w_v=rng.standard_normal((D, H, d_v)),
                w_g=rng.standard_normal((D, H, d_v)), w_o=rng.standard_normal((H, d_v, D_out)),
                gamma=np.array([0.9, 0.8, 0.99]), theta=rng.uniform(0.01, 1, d_k // 2))


def pin_block_projections_feed_the_core():
    """With one-hot projections (D = H·d_k = H·d_v, W_Q = W_K = W_V = the head's
    slice of the identity), q, k, v are the head slices of x; with w_g large
    the gate is the identity to 1e-12 and w_o the identity reassembles the
    heads, so the block equals GroupNorm of the core on the sliced x."""
    rng = np.random.default_rng(41)
    B, L, H, d = 2, 9, 3, 4
    x = rng.standard_normal((B, L, H * d))
    eye = np.eye(H * d).reshape(H * d, H, d)
    w_o = np.eye(H * d).reshape(H, d, H * d)
    g, th = np.array([0.9, 0.7, 0.99]), rng.uniform(0.01, 1, d // 2)
    # swish(c·1) with c = 60 is 60·σ(60) = 60 to 1e-24; GroupNorm removes the factor 60
    ones = np.zeros((H * d, H, d))
    z, _ = R.msr_block(np.concatenate([x, np.ones((B, L, 1))], -1),
                       np.concatenate([eye, np.zeros((1, H, d))], 0),
                       np.concatenate([eye, np.zeros((1, H, d))], 0),
                       np.concatenate([eye, np.zeros((1, H, d))], 0),
                       np.concatenate([ones, np.full((1, H, d), 60.0)], 0), w_o, g, th)
    xs = x.reshape(B, L, H, d).transpose(0, 2, 1, 3)
    o, _ = R.retention(xs, xs, xs, g, th)
    ref = 60.0 * R.group_norm(o)
    assert np.allclose(z, ref.transpose(0, 2, 1, 3).reshape(B, L, H * d), rtol=1e-12, atol=1e-10)


def pin_block_gate_and_projection():
    """swish(0) = 0 gives z = 0; z is linear in W_O; swish matches x·expit(x)."""
    p = _block_inputs(42)
    z0, _ = R.msr_block(**{**p, "w_g": np.zeros_like(p["w_g"])})
    assert np.all(z0 == 0.0)
    z1, _ = R.msr_block(**p)
    z2, _ = R.msr_block(**{**p, "w_o": 2.5 * p["w_o"]})
    assert np.allclose(z2, 2.5 * z1, rtol=1e-12, atol=1e-12)
    # one head, one gate column: compare against scipy's logistic function
    from scipy.special import expit
    o, _ = R.retention(np.einsum("bld,dhk->bhlk", p["x"], p["w_q"]),
                       np.einsum("bld,dhk->bhlk", p["x"], p["w_k"]),
                       np.einsum("bld,dhv->bhlv", p["x"], p["w_v"]), p["gamma"], p["theta"])
    y = R.group_norm(o)
    gp = np.einsum("bld,dhv->bhlv", p["x"], p["w_g"])
    ref = np.einsum("bhlv,hvo->blo", gp * expit(gp) * y, p["w_o"])
    assert np.allclose(z1, ref, rtol=1e-12, atol=1e-12)


def pin_block_groupnorm_removes_value_scale():
    """The core is linear in v, so scaling W_V by c > 0 scales every head's
    output by c, which GroupNorm with eps = 0 removes; the state scales by c."""
    p = _block_inputs(43)
    z1, s1 = R.msr_block(**p, gn_eps=0.0)
    z2, s2 = R.msr_block(**{**p, "w_v": 3.0 * p["w_v"]}, gn_eps=0.0)
    assert np.allclose(z1, z2, rtol=1e-10, atol=1e-10)
    assert np.allclose(s2, 3.0 * s1, rtol=1e-12, atol=1e-12)


PINS = [
    pin_demo_parallel_equals_recurrent, pin_rotation_fixed_angles, pin_retention_hand_case,
    pin_forms_match_brute_force, pin_linear_attention_limit, pin_gamma_zero, pin_single_token,
    pin_theta_zero_is_identity, pin_rotation_preserves_pair_norms, pin_position_shift_invariance,
    pin_exact_causality, pin_chunk_limits, pin_split_call, pin_ragged_tail, pin_linearity,
    pin_decode_steps_equal_recurrent, pin_groupnorm_matches_torch, pin_backward_finite_differences,
    pin_param_grads_finite_differences, pin_theta_grad_position_shift_invariance,
    pin_gamma_grad_single_token, pin_groupnorm_backward,
    pin_decay_row_sums_geometric_series, pin_normalised_gamma_one_is_a_running_mean,
    pin_normalised_cancels_under_groupnorm, pin_normalised_split_calls,
    pin_block_projections_feed_the_core, pin_block_gate_and_projection,
    pin_block_groupnorm_removes_value_scale,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ----------------------------------------------------------------------------
# Mutation test: every planted mistake must be caught by some pin.
# (function, text in its source, replacement) — applied to a copy of the
# oracle module's namespace, never to the file.
# ----------------------------------------------------------------------------

MUTANTS = {
    "rotation_sign": ("rotate_every_two", "out[..., 0::2] = -x[..., 1::2]", "out[..., 0::2] = x[..., 1::2]"),
    "rotation_halves": ("rotate_every_two",
                        "out[..., 0::2] = -x[..., 1::2]\n    out[..., 1::2] = x[..., 0::2]",
                        "h = x.shape[-1] // 2\n    out[..., :h] = -x[..., h:]\n    out[..., h:] = x[..., :h]"),
    "k_conjugate_angle": ("prologue", "kp = theta_shift(k, sin, cos)", "kp = theta_shift(k, -sin, cos)"),
    "no_scale": ("prologue", "/ math.sqrt(d_k)", ""),
    "scale_seq_len": ("prologue", "/ math.sqrt(d_k)", "/ math.sqrt(L)"),
    "mask_not_causal": ("decay_mask", "np.where(diff >= 0,", "np.where(diff >= -1,"),
    "mask_exponent_off_by_one": ("decay_mask", "np.maximum(diff, 0)", "np.maximum(diff - 1, 0)"),
    "parallel_state_decay": ("parallel_core", "np.arange(1, L + 1,", "np.arange(0, L,"),
    "recurrent_old_state_output": ("recurrent_core",
                                   "S = gb * S + kp[:, :, t, :, None] * v[:, :, t, None, :]\n        out[:, :, t] = np.einsum(\"bhk,bhkv->bhv\", qp[:, :, t], S)",
                                   "out[:, :, t] = np.einsum(\"bhk,bhkv->bhv\", qp[:, :, t], S)\n        S = gb * S + kp[:, :, t, :, None] * v[:, :, t, None, :]"),
    "chunk_xi": ("chunkwise_core", "np.arange(1, r + 1,", "np.arange(0, r,"),
    "chunk_zeta_reversed": ("chunkwise_core", "np.arange(r - 1, -1, -1,", "np.arange(0, r,"),
    "chunk_carry": ("chunkwise_core", "np.power(gh, float(r)) * S[:, h]", "np.power(gh, float(r - 1)) * S[:, h]"),
    "chunk_transposed_kv": ("chunkwise_core", "np.swapaxes(k_i * zeta[None, :, None], -1, -2) @ v_i",
                            "np.swapaxes(k_i[..., ::-1] * zeta[None, :, None], -1, -2) @ v_i"),
    "state_closed_form_power": ("state_closed_form", "np.power(g[h], float(L))", "np.power(g[h], float(L - 1))"),
    "gn_unbiased": ("group_norm", "((o - mu) ** 2).mean(axis=-1, keepdims=True)",
                    "((o - mu) ** 2).sum(axis=-1, keepdims=True) / (o.shape[-1] - 1)"),
    "gn_eps_outside": ("group_norm", "np.sqrt(var + float(eps))", "(np.sqrt(var) + float(eps))"),
    "decode_no_decay": ("decode_step", "S = g * state +", "S = state +"),
    "bwd_no_state_in_term": ("_rotated_grads", "dqp[:, h] += xi[None, :, None] * (dO[:, h] @",
                             "dqp[:, h] += 0.0 * xi[None, :, None] * (dO[:, h] @"),
    "bwd_adjoint_not_inverse": ("retention_backward", "dq = theta_shift(dqp, -sin, cos)",
                                "dq = theta_shift(dqp, sin, cos)"),
    "bwd_dk_untransposed": ("_rotated_grads", "np.swapaxes(G, -1, -2) @ qp[:, h]", "G @ qp[:, h]"),
    "bwd_dsin_power": ("_rotated_grads", "np.power(g[h], float(L)) * dSo", "np.power(g[h], float(L - 1)) * dSo"),
    "bwd_dk_no_scale": ("retention_backward", "/ math.sqrt(d_k)", ""),
    "pg_mask_derivative_power": ("retention_param_grads", "np.maximum(diff - 1.0, 0.0)", "np.maximum(diff, 0.0)"),
    "pg_xi_derivative": ("retention_param_grads", "dxi = (t + 1.0) * np.power(gh, t)", "dxi = t * np.power(gh, t)"),
    "pg_w_derivative": ("retention_param_grads", "e = L - 1.0 - t", "e = L - t"),
    "pg_sin_into_sout": ("retention_param_grads", "L * np.power(gh, L - 1.0)", "(L - 1.0) * np.power(gh, L - 1.0)"),
    "pg_theta_local_positions": ("retention_param_grads", "pos = t + int(pos0)", "pos = t"),
    "pg_theta_no_k_term": ("retention_param_grads", " + dkp * rotate_every_two(kp)", ""),
    "gnb_no_xhat_term": ("groupnorm_backward", " - xhat * (gw * xhat).mean(axis=-1, keepdims=True)", ""),
    "gnb_weight_not_applied": ("groupnorm_backward", "gw = d_y * w[None, :, None, :]", "gw = d_y"),
    "gnb_dweight_no_xhat": ("groupnorm_backward", "d_weight = (d_y * xhat).sum(axis=(0, 2))",
                            "d_weight = d_y.sum(axis=(0, 2))"),
    "rowsum_local_positions": ("decay_row_sums", "np.cumsum(terms)[int(pos0):]", "np.cumsum(terms)[:int(L)]"),
    "rowsum_off_by_one": ("decay_row_sums", "np.arange(n_max,", "np.arange(1, n_max + 1,"),
    "block_q_from_w_k": ("msr_block", 'q = np.einsum("bld,dhk->bhlk", x, _f64(w_q))',
                         'q = np.einsum("bld,dhk->bhlk", x, _f64(w_k))'),
    "block_sigmoid_gate": ("msr_block", "gate = gpre / (1.0 + np.exp(-gpre))", "gate = 1.0 / (1.0 + np.exp(-gpre))"),
    "block_gate_after_projection": ("msr_block", 'z = np.einsum("bhlv,hvo->blo", gate * y, _f64(w_o))',
                                    'z = np.einsum("bhlv,hvo->blo", y, _f64(w_o)) * gate.mean()'),
    "block_no_groupnorm": ("msr_block", "y = group_norm(o, gn_eps)", "y = o"),
    "normalised_state_unscaled": ("normalised_retention", "np.arange(1, L + 1, dtype=np.float64)) / r[h]",
                                  "np.arange(1, L + 1, dtype=np.float64))"),
}


def _make_mutant(name):
    import inspect
    import textwrap
    import types

    fn_name, old, new = MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(getattr(R, fn_name)))
    assert old in src, f"mutant {name}: pattern not found in {fn_name}"
    src = src.replace(old, new, 1)
    mod = types.ModuleType("oracle_mutant")
    mod.__dict__.update({k: v for k, v in R.__dict__.items() if not k.startswith("__")})
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    # functions defined in the copy must see the mutated function
    for k, v in list(mod.__dict__.items()):
        if isinstance(v, types.FunctionType) and v.__module__ == R.__name__:
            mod.__dict__[k] = types.FunctionType(v.__code__, mod.__dict__, v.__name__, v.__defaults__)
    mod.__dict__[fn_name] = types.FunctionType(
        mod.__dict__[fn_name].__code__, mod.__dict__, fn_name, mod.__dict__[fn_name].__defaults__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, monkeypatch):
    mod = _make_mutant(name)
    global R
    saved = R
    R = mod
    caught = []
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError, FloatingPointError, IndexError):
                caught.append(pin.__name__)
    finally:
        R = saved
    assert caught, f"mutant {name} was not caught by any pin"


# ------------------------------------------------------------- backward --
@pytest.mark.parametrize("with_state,with_dso,pos0", [(False, False, 0), (True, False, 3), (True, True, 11)])
def test_backward_matches_finite_differences(with_state, with_dso, pos0):
    _backward_fd_check(with_state, with_dso, pos0)
