"""Float64 CPU oracle for RetNet multi-scale retention (MSR).

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code,
constants or helpers with the CUDA path.

Sources (web pages about RetNet; formulas partly garbled by extraction):

* [P1] «从RoPE到Retention：一文拆解RetNet如何用'旋转'和'衰减'重塑序列建模»
  (jsqmd.com news 854720): §2 (theta_shift / rotate_every_two, Q←Q⊙Θ,
  K←K⊙Θ̄), §3 (decay D_nm), §4.1 parallel form, §4.2 recurrent form
  S_n = γS_{n-1} + K_nᵀV_n, output Q_nS_n, §4.3 chunkwise form, §5 (GroupNorm,
  division by √d, zero initial state of shape heads×d×d).
* [P3] RetNet 保留网络 explainer (aiqz.cc article retnet-network):
  "核心机制" (mask M_nj = γ^{n-j} for n ≥ j, 0 for n < j), "并行表征"
  ((QKᵀ⊙M)V without softmax), "循环表征" (decay the state by γ, add the outer
  product K_nᵀV_n, read with Q_n), "分块循环" (parallel inside a chunk, γ^b
  carry between chunks, b=1 → recurrent, b=n → parallel), "Python 演示"
  (parallel and recurrent agree to < 1e-8), "常见误区" (the factorisation
  γ^{n-j} = γ^n·γ^{-j} turns the pairwise sum into a state recurrence).
* [P4] «RetNet：Transformer的革命性继任者？» (project page of a PyTorch
  implementation): SimpleRetention with W_Q, W_K, W_V applied to the input X;
  MultiScaleRetention as one SimpleRetention per head in parallel.
* [P5] «Transformer后繼有模！MSRA提出全新大模型基礎架構» (b99b.cn): GroupNorm
  is used for its scale invariance; complex-valued position encoding.

Readings taken where the pages are silent or garbled (each is listed again in
the design notes):

R1  rotate_every_two acts on interleaved pairs (2i, 2i+1) and maps
    (a, b) → (−b, a); theta_shift(x) = x·cos + rotate_every_two(x)·sin with the
    angle n·θ_i shared by both members of pair i.  So each pair is rotated
    counter-clockwise by n·θ_i.
R2  Q and K are both rotated by +n·θ at their own absolute position n.  The
    real dot product then depends on the position difference only, which is
    what the complex-conjugate pairing Θ / Θ̄ of [P1] §2 expresses.
R3  Exactly one score scale d_k^{-1/2} is applied, folded into K′ ([P1] §5
    "除以√d"; the `/ seq_len.sqrt()` of the [P1] §4.1 snippet is read as a
    garbled √d).
R4  state_in is the state *before* the first token (S_{-1}); its contribution
    to token t decays by γ^{t+1}.
R5  A decode step outputs q′·S_n with the *updated* state ([P1] §4.2
    "Output = QₙSₙ"; [P3] "循环表征").
R6  Masked entries (n < m) are exact zeros.
R7  GroupNorm: one group per head over the d_v channels of one token,
    biased variance, eps given by the caller (1e-5 default), optional affine.
R8  A ragged last chunk of length r uses carry γ^r and ζ_j = γ^{r-1-j}.
R10 The MSR block around the core (the projections of [P4]'s SimpleRetention,
    q = X·W_Q, k = X·W_K, v = X·W_V per head; heads in parallel, outputs
    concatenated; per-head GroupNorm of [P1] §5).  The pages give no output
    projection or gate; the block takes the published RetNet MSR
    definition for them: Z = (swish(X·W_G) ⊙ concat_h GN(O_h))·W_O with
    swish(x) = x·σ(x).
R9  The row-normalised decay of [P1] §5 ("三重标准化": the √d division, the
    decay weights normalised per row, a global scaling): row N of D is
    divided by its sum over the absolute positions 0..N it covers,
    r_N = Σ_{i=0}^{N} γ^i, the state term standing for the positions before
    pos0 (so split calls agree); the global scaling has no stated value and is
    1.  With GroupNorm after it, the whole normalisation cancels up to eps
    (the scale invariance of [P5]).

Conventions: q, k are [B, H, L, d_k]; v is [B, H, L, d_v]; gamma is [H];
theta is [d_k/2]; states are [B, H, d_k, d_v]; absolute position of local
index t is n = pos0 + t.  Every function computes in float64.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "rotate_every_two",
    "theta_shift",
    "rotation_tables",
    "prologue",
    "decay_mask",
    "parallel_core",
    "recurrent_core",
    "chunkwise_core",
    "state_closed_form",
    "retention",
    "retention_backward",
    "retention_param_grads",
    "groupnorm_backward",
    "decay_row_sums",
    "normalised_retention",
    "msr_block",
    "decode_step",
    "group_norm",
    "brute_force",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# Θ rotation prologue ([P1] §2; readings R1–R3)
# --------------------------------------------------------------------------

def rotate_every_two(x):
    """(x_{2i}, x_{2i+1}) → (−x_{2i+1}, x_{2i}) on the last axis ([P1] §2, R1)."""
    x = _f64(x)
    out = np.empty_like(x)
    out[..., 0::2] = -x[..., 1::2]
    out[..., 1::2] = x[..., 0::2]
    return out


def rotation_tables(positions, theta):
    """sin/cos of n·θ_i, each value repeated for both members of pair i.

    positions: int array [L]; theta: [d/2].  Returns (sin, cos) of shape [L, d].
    """
    n = np.asarray(positions, dtype=np.float64)[:, None]
    ang = n * _f64(theta)[None, :]
    return np.repeat(np.sin(ang), 2, axis=-1), np.repeat(np.cos(ang), 2, axis=-1)


def theta_shift(x, sin, cos):
    """x·cos + rotate_every_two(x)·sin ([P1] §2)."""
    x = _f64(x)
    return x * cos + rotate_every_two(x) * sin


def prologue(q, k, theta, pos0=0):
    """q′ = Θ-rotated q; k′ = d_k^{-1/2}·Θ-rotated k (R2, R3)."""
    q = _f64(q)
    k = _f64(k)
    L, d_k = q.shape[-2], q.shape[-1]
    sin, cos = rotation_tables(np.arange(L) + int(pos0), theta)
    qp = theta_shift(q, sin, cos)
    kp = theta_shift(k, sin, cos) / math.sqrt(d_k)
    return qp, kp


# --------------------------------------------------------------------------
# Core forms on already-rotated q′, k′ (per head; broadcast over B, H)
# --------------------------------------------------------------------------

def decay_mask(gamma, L):
    """D_nm = γ^{n−m} for n ≥ m, exactly 0 otherwise ([P1] §3; [P3] 核心机制, R6)."""
    n = np.arange(L)[:, None]
    m = np.arange(L)[None, :]
    diff = n - m
    with np.errstate(divide="ignore", invalid="ignore"):
        # γ^0 = 1 also for γ = 0; entries above the diagonal are set to 0.
        d = np.where(diff >= 0, np.power(float(gamma), np.maximum(diff, 0).astype(np.float64)), 0.0)
    return d


def _heads(gamma, H):
    g = _f64(gamma).reshape(-1)
    if g.shape[0] != H:
        raise ValueError("gamma must have one value per head")
    return g


def parallel_core(qp, kp, v, gamma, state_in=None):
    """O = (Q′K′ᵀ ⊙ D)V + γ^{t+1} q′_t S_in, and S_out ([P1] §4.1; [P3] 并行表征, R4)."""
    qp, kp, v = _f64(qp), _f64(kp), _f64(v)
    B, H, L, _ = qp.shape
    g = _heads(gamma, H)
    out = np.zeros(v.shape[:-2] + (L, v.shape[-1]))
    for h in range(H):
        D = decay_mask(g[h], L)
        scores = qp[:, h] @ np.swapaxes(kp[:, h], -1, -2)
        out[:, h] = (scores * D) @ v[:, h]
        if state_in is not None:
            xi = np.power(g[h], np.arange(1, L + 1, dtype=np.float64))
            out[:, h] += xi[None, :, None] * (qp[:, h] @ _f64(state_in)[:, h])
    return out, state_closed_form(kp, v, gamma, state_in)


def state_closed_form(kp, v, gamma, state_in=None):
    """S_out = γ^L S_in + Σ_m γ^{L−1−m} k′_mᵀ v_m (the recurrence of [P1] §4.2 unrolled)."""
    kp, v = _f64(kp), _f64(v)
    B, H, L, d_k = kp.shape
    g = _heads(gamma, H)
    S = np.zeros((B, H, d_k, v.shape[-1]))
    for h in range(H):
        w = np.power(g[h], np.arange(L - 1, -1, -1, dtype=np.float64))
        S[:, h] = np.swapaxes(kp[:, h] * w[None, :, None], -1, -2) @ v[:, h]
        if state_in is not None:
            S[:, h] += np.power(g[h], float(L)) * _f64(state_in)[:, h]
    return S


def recurrent_core(qp, kp, v, gamma, state_in=None):
    """S_n = γS_{n−1} + k′_nᵀv_n ; o_n = q′_n S_n ([P1] §4.2; [P3] 循环表征, R5)."""
    qp, kp, v = _f64(qp), _f64(kp), _f64(v)
    B, H, L, d_k = qp.shape
    d_v = v.shape[-1]
    g = _heads(gamma, H)
    S = np.zeros((B, H, d_k, d_v)) if state_in is None else _f64(state_in).copy()
    out = np.zeros((B, H, L, d_v))
    gb = g[None, :, None, None]
    for t in range(L):
        S = gb * S + kp[:, :, t, :, None] * v[:, :, t, None, :]
        out[:, :, t] = np.einsum("bhk,bhkv->bhv", qp[:, :, t], S)
    return out, S


def chunkwise_core(qp, kp, v, gamma, state_in=None, chunk=None):
    """Chunkwise recurrent form ([P1] §4.3; [P3] 分块循环; R8 for a ragged tail).

    Within chunk i (local index j = 0..r−1, r ≤ chunk) and with S the state
    at the end of chunk i−1:
        o_j   = γ^{j+1} q′_j S + Σ_{m ≤ j} γ^{j−m} (q′_j·k′_m) v_m
        S_new = γ^r S + Σ_j γ^{r−1−j} k′_jᵀ v_j
    These follow from unrolling S_n = γS_{n−1} + k′_nᵀv_n over one chunk
    (the γ^{n−j} = γ^n·γ^{−j} factorisation of [P3] 常见误区).
    """
    qp, kp, v = _f64(qp), _f64(kp), _f64(v)
    B, H, L, d_k = qp.shape
    d_v = v.shape[-1]
    g = _heads(gamma, H)
    if chunk is None:
        chunk = L
    if chunk < 1:
        raise ValueError("chunk must be >= 1")
    S = np.zeros((B, H, d_k, d_v)) if state_in is None else _f64(state_in).copy()
    out = np.zeros((B, H, L, d_v))
    for start in range(0, L, chunk):
        r = min(chunk, L - start)
        sl = slice(start, start + r)
        for h in range(H):
            gh = g[h]
            xi = np.power(gh, np.arange(1, r + 1, dtype=np.float64))        # γ^{j+1}
            zeta = np.power(gh, np.arange(r - 1, -1, -1, dtype=np.float64))  # γ^{r−1−j}
            D = decay_mask(gh, r)
            q_i, k_i, v_i = qp[:, h, sl], kp[:, h, sl], v[:, h, sl]
            inner = ((q_i @ np.swapaxes(k_i, -1, -2)) * D) @ v_i
            cross = xi[None, :, None] * (q_i @ S[:, h])
            out[:, h, sl] = inner + cross
            S[:, h] = np.power(gh, float(r)) * S[:, h] + np.swapaxes(k_i * zeta[None, :, None], -1, -2) @ v_i
    return out, S


# --------------------------------------------------------------------------
# GroupNorm epilogue ([P1] §5; [P5]; reading R7)
# --------------------------------------------------------------------------

def group_norm(o, eps=1e-5, weight=None, bias=None):
    """Normalise each (b, h, t) row over its d_v channels; optional affine of shape [H, d_v]."""
    o = _f64(o)
    mu = o.mean(axis=-1, keepdims=True)
    var = ((o - mu) ** 2).mean(axis=-1, keepdims=True)
    y = (o - mu) / np.sqrt(var + float(eps))
    if weight is not None:
        y = y * _f64(weight)[None, :, None, :]
    if bias is not None:
        y = y + _f64(bias)[None, :, None, :]
    return y


def groupnorm_backward(o, d_y, eps=1e-5, weight=None):
    """Gradients of ``group_norm`` (R7) for the upstream gradient d_y of its
    output.  Returns (d_o, d_weight, d_bias); d_weight and d_bias have the
    affine's shape [H, d_v] and sum over batch and tokens (weight None means
    ones).  Per row, over its N = d_v channels, with μ the mean, var the
    biased variance, σ = √(var + eps), x̂ = (o − μ)/σ and g = d_y ⊙ weight,
    differentiating y = x̂·weight + bias through μ and var (both depend on
    every channel of the row):
      d_o      = (g − mean(g) − x̂·mean(g ⊙ x̂)) / σ
      d_weight = Σ_rows d_y ⊙ x̂,   d_bias = Σ_rows d_y
    """
    o, d_y = _f64(o), _f64(d_y)
    H, d_v = o.shape[1], o.shape[-1]
    w = np.ones((H, d_v)) if weight is None else _f64(weight)
    mu = o.mean(axis=-1, keepdims=True)
    var = ((o - mu) ** 2).mean(axis=-1, keepdims=True)
    sigma = np.sqrt(var + float(eps))
    xhat = (o - mu) / sigma
    gw = d_y * w[None, :, None, :]
    d_o = (gw - gw.mean(axis=-1, keepdims=True) - xhat * (gw * xhat).mean(axis=-1, keepdims=True)) / sigma
    d_weight = (d_y * xhat).sum(axis=(0, 2))
    d_bias = d_y.sum(axis=(0, 2))
    return d_o, d_weight, d_bias


# --------------------------------------------------------------------------
# Full operation and the decode step
# --------------------------------------------------------------------------

def retention(q, k, v, gamma, theta, pos0=0, state_in=None, form="chunkwise",
              chunk=None, gn=None):
    """Prologue + one of the three forms + optional GroupNorm.

    Returns (out, state_out).  ``gn`` is None or a dict with keys eps, weight,
    bias (weight/bias may be None).
    """
    qp, kp = prologue(q, k, theta, pos0)
    if form == "parallel":
        out, S = parallel_core(qp, kp, v, gamma, state_in)
    elif form == "recurrent":
        out, S = recurrent_core(qp, kp, v, gamma, state_in)
    elif form == "chunkwise":
        out, S = chunkwise_core(qp, kp, v, gamma, state_in, chunk)
    else:
        raise ValueError(form)
    if gn is not None:
        out = group_norm(out, gn.get("eps", 1e-5), gn.get("weight"), gn.get("bias"))
    return out, S


def decay_row_sums(gamma, pos0, L):
    """r[h, t] = Σ_{i=0}^{N} γ_h^i with N = pos0 + t: the sum of row N of the
    decay mask over every position it covers (R9), summed term by term."""
    g = _f64(gamma).reshape(-1)
    n_max = int(pos0) + int(L)
    r = np.empty((g.shape[0], int(L)))
    for h in range(g.shape[0]):
        terms = np.power(g[h], np.arange(n_max, dtype=np.float64))   # γ^0 … γ^{N_max}
        r[h] = np.cumsum(terms)[int(pos0):]
    return r


def normalised_retention(q, k, v, gamma, theta, pos0=0, state_in=None, gn=None):
    """Retention with the row-normalised decay D̃ of [P1] §5 (R9), parallel
    form: out = (Q′K′ᵀ ⊙ D̃)V + (ξ/r) ⊙ (Q′ S_in) with D̃_tm = D_tm / r_t and
    ξ_t = γ^{t+1}, then the optional GroupNorm.  Returns out only (the state
    is not affected by the normalisation)."""
    qp, kp = prologue(q, k, theta, pos0)
    v = _f64(v)
    B, H, L, _ = qp.shape
    g = _heads(gamma, H)
    r = decay_row_sums(g, pos0, L)
    out = np.zeros((B, H, L, v.shape[-1]))
    for h in range(H):
        Dn = decay_mask(g[h], L) / r[h][:, None]
        out[:, h] = ((qp[:, h] @ np.swapaxes(kp[:, h], -1, -2)) * Dn) @ v[:, h]
        if state_in is not None:
            xi = np.power(g[h], np.arange(1, L + 1, dtype=np.float64)) / r[h]
            out[:, h] += xi[None, :, None] * (qp[:, h] @ _f64(state_in)[:, h])
    if gn is not None:
        out = group_norm(out, gn.get("eps", 1e-5), gn.get("weight"), gn.get("bias"))
    return out


def msr_block(x, w_q, w_k, w_v, w_g, w_o, gamma, theta, pos0=0, state_in=None,
              gn_eps=1e-5, chunk=None):
    """The MSR block around the core (R10): x [B, L, D]; w_q, w_k [D, H, d_k];
    w_v, w_g [D, H, d_v]; w_o [H, d_v, D_out].  Per head q = x·W_Q, k = x·W_K,
    v = x·W_V ([P4]), the chunkwise core with the prologue, GroupNorm per
    head ([P1] §5), the swish gate and the output projection.  Returns
    (z [B, L, D_out], state_out)."""
    x = _f64(x)
    q = np.einsum("bld,dhk->bhlk", x, _f64(w_q))
    k = np.einsum("bld,dhk->bhlk", x, _f64(w_k))
    v = np.einsum("bld,dhv->bhlv", x, _f64(w_v))
    o, S = retention(q, k, v, gamma, theta, pos0, state_in, "chunkwise", chunk)
    y = group_norm(o, gn_eps)
    gpre = np.einsum("bld,dhv->bhlv", x, _f64(w_g))
    gate = gpre / (1.0 + np.exp(-gpre))                               # swish(x) = x·σ(x)
    z = np.einsum("bhlv,hvo->blo", gate * y, _f64(w_o))
    return z, S


def _rotated_grads(q, k, v, gamma, theta, pos0=0, state_in=None, d_out=None,
                   d_state_out=None):
    """The chain rule applied to the parallel form with the state terms
    ([P1] §4.1, R4), per head with A = D (the causal decay mask),
    ξ_t = γ^{t+1} and w_m = γ^{L−1−m}:
      out    = (Q′K′ᵀ ⊙ A) V + ξ ⊙ (Q′ S_in)
      S_out  = γ^L S_in + Σ_m w_m k′_mᵀ v_m
    give, with G = (dO Vᵀ) ⊙ A,
      dV     = (Q′K′ᵀ ⊙ A)ᵀ dO + (w ⊙ K′) dS_out
      dQ′    = G K′ + ξ ⊙ (dO S_inᵀ)
      dK′    = Gᵀ Q′ + (w ⊙ V) dS_outᵀ
      dS_in  = (ξ ⊙ Q′)ᵀ dO + γ^L dS_out
    Returns (q′, k′, dQ′, dK′, dV, dS_in): the gradients with respect to the
    rotated operands, before the prologue's adjoint."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d_k = q.shape
    d_v = v.shape[-1]
    g = _heads(gamma, H)
    qp, kp = prologue(q, k, theta, pos0)
    dO = _f64(d_out)
    dqp = np.zeros_like(qp)
    dkp = np.zeros_like(kp)
    dv = np.zeros_like(v)
    dS_in = np.zeros((B, H, d_k, d_v))
    for h in range(H):
        A = decay_mask(g[h], L)
        P = (qp[:, h] @ np.swapaxes(kp[:, h], -1, -2)) * A            # scores with decay
        G = (dO[:, h] @ np.swapaxes(v[:, h], -1, -2)) * A
        xi = np.power(g[h], np.arange(1, L + 1, dtype=np.float64))
        w = np.power(g[h], np.arange(L - 1, -1, -1, dtype=np.float64))
        dv[:, h] = np.swapaxes(P, -1, -2) @ dO[:, h]
        dqp[:, h] = G @ kp[:, h]
        dkp[:, h] = np.swapaxes(G, -1, -2) @ qp[:, h]
        dS_in[:, h] = np.swapaxes(xi[None, :, None] * qp[:, h], -1, -2) @ dO[:, h]
        if state_in is not None:
            dqp[:, h] += xi[None, :, None] * (dO[:, h] @ np.swapaxes(_f64(state_in)[:, h], -1, -2))
        if d_state_out is not None:
            dSo = _f64(d_state_out)[:, h]
            dv[:, h] += (w[None, :, None] * kp[:, h]) @ dSo
            dkp[:, h] += (w[None, :, None] * v[:, h]) @ np.swapaxes(dSo, -1, -2)
            dS_in[:, h] += np.power(g[h], float(L)) * dSo
    return qp, kp, dqp, dkp, dv, dS_in


def retention_backward(q, k, v, gamma, theta, pos0=0, state_in=None, d_out=None,
                       d_state_out=None):
    """Gradients of ``retention`` (no GroupNorm) with respect to q, k, v and
    state_in, for the upstream gradients d_out (of out) and d_state_out (of
    state_out, or None).  Returns (dq, dk, dv, d_state_in).

    dQ′, dK′, dV and dS_in come from the chain rule through the parallel
    form (``_rotated_grads``); then through the prologue (R1-R3: q′ = R q,
    k′ = d_k^{-1/2} R k with R an orthogonal rotation per position)
    dq = Rᵀ dQ′, dk = d_k^{-1/2} Rᵀ dK′, Rᵀ being the rotation by −n·θ.
    """
    _, _, dqp, dkp, dv, dS_in = _rotated_grads(q, k, v, gamma, theta, pos0, state_in, d_out,
                                               d_state_out)
    L, d_k = dqp.shape[-2], dqp.shape[-1]
    sin, cos = rotation_tables(np.arange(L) + int(pos0), theta)
    dq = theta_shift(dqp, -sin, cos)                                   # Rᵀ = rotation by −nθ
    dk = theta_shift(dkp, -sin, cos) / math.sqrt(d_k)
    return dq, dk, dv, dS_in


def retention_param_grads(q, k, v, gamma, theta, pos0=0, state_in=None, d_out=None,
                          d_state_out=None):
    """Gradients of ``retention`` (no GroupNorm) with respect to the decay
    rates γ [H] and the rotation frequencies θ [d_k/2], for the same
    upstream gradients as ``retention_backward``.  Returns (d_gamma, d_theta).

    [P1] §2 makes θ a learnable parameter; γ is set per head at
    initialisation ([P1] §3) and is differentiated too, for callers that
    learn it.  The gradients sum over the batch (and d_theta over the heads).

    d_gamma: every γ-dependent factor of the parallel form with the state
    terms (R4) is differentiated and contracted with what it multiplies:
      ∂D_nm/∂γ = (n−m)·γ^{n−m−1}   below the diagonal (0 on and above it)
      ∂ξ_t/∂γ  = (t+1)·γ^t          the state_in term of token t
      ∂w_m/∂γ  = (L−1−m)·γ^{L−2−m}  key m's share of state_out
      ∂γ^L/∂γ  = L·γ^{L−1}           state_in's share of state_out
    d_theta: through the prologue.  Pair i of q′_t is pair i of q_t rotated
    by the angle (pos0+t)·θ_i, so ∂q′_t/∂θ_i is (pos0+t)·rotate_every_two(q′_t)
    on that pair and zero elsewhere; the same holds for k′_t (the 1/√d_k
    scale rides along).  Both are contracted with dQ′, dK′.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, L, d_k = q.shape
    g = _heads(gamma, H)
    qp, kp, dqp, dkp, _, _ = _rotated_grads(q, k, v, gamma, theta, pos0, state_in, d_out,
                                            d_state_out)
    dO = _f64(d_out)
    diff = (np.arange(L)[:, None] - np.arange(L)[None, :]).astype(np.float64)
    t = np.arange(L, dtype=np.float64)
    d_gamma = np.zeros(H)
    for h in range(H):
        gh = g[h]
        dD = np.where(diff > 0, diff * np.power(gh, np.maximum(diff - 1.0, 0.0)), 0.0)
        scores = qp[:, h] @ np.swapaxes(kp[:, h], -1, -2)              # q′_n · k′_m
        dov = dO[:, h] @ np.swapaxes(v[:, h], -1, -2)                  # dO_n · v_m
        d_gamma[h] = np.sum(scores * dov * dD[None])
        if state_in is not None:
            S0 = _f64(state_in)[:, h]
            dxi = (t + 1.0) * np.power(gh, t)
            d_gamma[h] += np.sum(dxi[None, :, None] * (qp[:, h] @ S0) * dO[:, h])
        if d_state_out is not None:
            dSo = _f64(d_state_out)[:, h]
            e = L - 1.0 - t                                            # exponent of w_m
            dw = np.where(e > 0, e * np.power(gh, np.maximum(e - 1.0, 0.0)), 0.0)
            d_gamma[h] += np.einsum("m,bmk,bmv,bkv->", dw, kp[:, h], v[:, h], dSo)
            if state_in is not None:
                d_gamma[h] += L * np.power(gh, L - 1.0) * np.sum(dSo * _f64(state_in)[:, h])
    pos = t + int(pos0)
    per_elem = pos[None, None, :, None] * (dqp * rotate_every_two(qp) + dkp * rotate_every_two(kp))
    d_theta = per_elem[..., 0::2].sum(axis=(0, 1, 2)) + per_elem[..., 1::2].sum(axis=(0, 1, 2))
    return d_gamma, d_theta


def decode_step(q, k, v, gamma, theta, pos, state, gn=None):
    """One recurrent step at absolute position ``pos`` ([P1] §4.2, R5).

    q, k: [B, H, d_k]; v: [B, H, d_v]; state: [B, H, d_k, d_v].
    Returns (o [B, H, d_v], new_state).
    """
    q, k, v, state = _f64(q), _f64(k), _f64(v), _f64(state)
    qp, kp = prologue(q[:, :, None, :], k[:, :, None, :], theta, pos)
    qp, kp = qp[:, :, 0], kp[:, :, 0]
    g = _heads(gamma, q.shape[1])[None, :, None, None]
    S = g * state + kp[..., :, None] * v[..., None, :]
    o = np.einsum("bhk,bhkv->bhv", qp, S)
    if gn is not None:
        o = group_norm(o[:, :, None, :], gn.get("eps", 1e-5), gn.get("weight"), gn.get("bias"))[:, :, 0]
    return o, S


# --------------------------------------------------------------------------
# Brute force: the definition written out with scalar loops (tiny inputs)
# --------------------------------------------------------------------------

def brute_force(q, k, v, gamma, theta, pos0=0, state_in=None):
    """Scalar-loop evaluation of out and state_out straight from the definitions.

    Rotation uses math.cos / math.sin per pair; the output is the double sum
    Σ_{m ≤ t} γ^{t−m} (q′_t·k′_m) v_m plus γ^{t+1} q′_t S_in, and the state is
    γ^L S_in + Σ_m γ^{L−1−m} k′_mᵀ v_m.  Pure Python: tiny shapes only.
    """
    q = np.asarray(q, dtype=np.float64).tolist()
    k = np.asarray(k, dtype=np.float64).tolist()
    v = np.asarray(v, dtype=np.float64).tolist()
    th = [float(t) for t in np.asarray(theta, dtype=np.float64)]
    gam = [float(x) for x in np.asarray(gamma, dtype=np.float64)]
    S_in = None if state_in is None else np.asarray(state_in, dtype=np.float64).tolist()
    B, H, L, d_k = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    d_v = len(v[0][0][0])
    scale = 1.0 / math.sqrt(d_k)

    def rot(x, n):
        y = [0.0] * d_k
        for i in range(d_k // 2):
            c, s = math.cos(n * th[i]), math.sin(n * th[i])
            a, b = x[2 * i], x[2 * i + 1]
            y[2 * i] = a * c - b * s
            y[2 * i + 1] = b * c + a * s
        return y

    out = [[[[0.0] * d_v for _ in range(L)] for _ in range(H)] for _ in range(B)]
    st = [[[[0.0] * d_v for _ in range(d_k)] for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            g = gam[h]
            qr = [rot(q[b][h][t], pos0 + t) for t in range(L)]
            kr = [[scale * e for e in rot(k[b][h][t], pos0 + t)] for t in range(L)]
            for t in range(L):
                acc = [0.0] * d_v
                for m in range(t + 1):
                    w = (g ** (t - m)) * sum(qr[t][c] * kr[m][c] for c in range(d_k))
                    for c in range(d_v):
                        acc[c] += w * v[b][h][m][c]
                if S_in is not None:
                    gt = g ** (t + 1)
                    for c in range(d_v):
                        acc[c] += gt * sum(qr[t][kk] * S_in[b][h][kk][c] for kk in range(d_k))
                out[b][h][t] = acc
            for kk in range(d_k):
                for c in range(d_v):
                    s = 0.0 if S_in is None else (g ** L) * S_in[b][h][kk][c]
                    for m in range(L):
                        s += (g ** (L - 1 - m)) * kr[m][kk] * v[b][h][m][c]
                    st[b][h][kk][c] = s
    return np.array(out), np.array(st)
