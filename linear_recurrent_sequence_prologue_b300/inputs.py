"""Seeded synthetic inputs for the retention workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
only draws random numbers and builds the per-head / per-pair parameter
vectors; it holds none of the retention arithmetic.

Workloads (shapes of the MSR core at the model sizes the RetNet pages
discuss; the 512-hidden / 8-head shape is the example model of «RetNet：
Transformer的革命性继任者？», the 7B / 8k point is the headline of
«Transformer后繼有模！MSRA提出全新大模型基礎架構»):

* ``tiny``     B1 H2 L64 d_k=d_v=16, fp32, chunk 16, q,k,v ~ N(0,1)
* ``small``    B4 H8 L2048 d_k=d_v=64, bf16, chunk 64, q,k,v ~ N(0,1)/√64
* ``msr1p3b``  B8 H8 L2048 d_k256 d_v512, bf16, chunk 128,
               q,k,v ~ N(0, (0.02·√2048)²), per-head GroupNorm
* ``msr7b``    B2 H16 L8192 d_k256 d_v512, bf16, chunk 128,
               q,k,v ~ N(0, (0.02·√4096)²), state_in ~ N(0, 1e-2)
* ``decode``   batch 128 H16 d_k256 d_v512, fp32 state ~ N(0, 1e-2),
               q,k,v ~ N(0,1)/16 per token, 1024 steps

Decay per head γ_h = 1 − 2^(−5−h); rotation frequencies
θ_i = 10000^(−2i/d_k).  Draw order: q, k, v, state_in, all in fp32 from one
``torch.Generator`` seeded with ``seed``, then cast to the workload dtype.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d_k: int
    d_v: int
    dtype: str          # "f32" or "bf16" (inputs and outputs)
    chunk: int
    qkv_std: float
    state_std: float = 0.0   # 0 → no state_in (zero initial state)
    groupnorm: bool = False
    gn_eps: float = 1e-5
    steps: int = 0           # decode only: number of sequential steps
    notes: str = ""

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 64, 16, 16, "f32", 16, 1.0),
    "small": Workload("small", 4, 8, 2048, 64, 64, "bf16", 64, 1.0 / math.sqrt(64)),
    "msr1p3b": Workload("msr1p3b", 8, 8, 2048, 256, 512, "bf16", 128,
                        0.02 * math.sqrt(2048), groupnorm=True),
    "msr7b": Workload("msr7b", 2, 16, 8192, 256, 512, "bf16", 128,
                      0.02 * math.sqrt(4096), state_std=0.1,
                      notes="q,k,v std 0.02*sqrt(hidden=4096) (same recipe as msr1p3b)"),
    "decode": Workload("decode", 128, 16, 1, 256, 512, "bf16", 1, 1.0 / 16,
                       state_std=0.1, steps=1024),
}


def gamma_schedule(H: int) -> np.ndarray:
    """γ_h = 1 − 2^(−5−h) as float32 (exact for h ≤ 18)."""
    return np.array([1.0 - 2.0 ** (-5 - h) for h in range(H)], dtype=np.float32)


def theta_schedule(d_k: int) -> np.ndarray:
    """θ_i = 10000^(−2i/d_k), i = 0 .. d_k/2 − 1, as float32."""
    i = np.arange(d_k // 2, dtype=np.float64)
    return np.power(10000.0, -2.0 * i / d_k).astype(np.float32)


def _randn(gen, shape, std):
    return torch.randn(*shape, generator=gen, dtype=torch.float32) * std


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw q, k, v (and state_in) for a sequence workload on the CPU.

    Returns a dict of CPU tensors in the workload dtype (state in fp32) plus
    the γ and θ vectors as float32 numpy arrays.
    """
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q = _randn(gen, (w.B, w.H, w.L, w.d_k), w.qkv_std).to(w.torch_dtype)
    k = _randn(gen, (w.B, w.H, w.L, w.d_k), w.qkv_std).to(w.torch_dtype)
    v = _randn(gen, (w.B, w.H, w.L, w.d_v), w.qkv_std).to(w.torch_dtype)
    state = None
    if w.state_std > 0:
        state = _randn(gen, (w.B, w.H, w.d_k, w.d_v), w.state_std)
    return {
        "q": q, "k": k, "v": v, "state_in": state,
        "gamma": gamma_schedule(w.H), "theta": theta_schedule(w.d_k),
    }


def make_grad_inputs(w: Workload, seed: int = 1, d_out_std: float = 1.0,
                     d_state_std: float = 0.0) -> dict:
    """Upstream gradients for the gradient pass: d_out [B, H, L, d_v] in the
    workload dtype and (when d_state_std > 0) d_state_out [B, H, d_k, d_v]
    fp32, both N(0, std²) on the CPU."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    d_out = _randn(gen, (w.B, w.H, w.L, w.d_v), d_out_std).to(w.torch_dtype)
    d_state = _randn(gen, (w.B, w.H, w.d_k, w.d_v), d_state_std) if d_state_std > 0 else None
    return {"d_out": d_out, "d_state_out": d_state}


def make_decode_inputs(w: Workload, seed: int = 0, steps: int | None = None,
                       device: str = "cpu") -> dict:
    """Initial state and per-step q, k, v for the decode workload.

    q, k: [steps, B, H, d_k]; v: [steps, B, H, d_v]; state: [B, H, d_k, d_v].
    ``device='cuda'`` draws on the GPU with a seeded CUDA generator (used by the
    benchmark, where the CPU draw of ~4 GB would dominate the run).
    """
    steps = w.steps if steps is None else steps
    gen = torch.Generator(device=device).manual_seed(seed)

    def rn(shape, std):
        return torch.randn(*shape, generator=gen, dtype=torch.float32, device=device) * std

    q = rn((steps, w.B, w.H, w.d_k), w.qkv_std).to(w.torch_dtype)
    k = rn((steps, w.B, w.H, w.d_k), w.qkv_std).to(w.torch_dtype)
    v = rn((steps, w.B, w.H, w.d_v), w.qkv_std).to(w.torch_dtype)
    state = rn((w.B, w.H, w.d_k, w.d_v), w.state_std)
    return {"q": q, "k": k, "v": v, "state": state,
            "gamma": gamma_schedule(w.H), "theta": theta_schedule(w.d_k)}


def to_f64(t) -> np.ndarray:
    """Exact float64 copy of what the GPU sees (bf16 and fp32 embed exactly)."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
