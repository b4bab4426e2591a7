"""GPU parity: every ABI call against the float64 oracle on seeded inputs.

Ordered from small to large.  Sizes the oracle finishes in seconds span
several tiles and a ragged tail; the full workloads are checked on sampled
(b, h) pairs, which the oracle computes head by head.
"""

import numpy as np
import pytest
import torch

import linear_recurrent_sequence_prologue_b300 as R
from linear_recurrent_sequence_prologue_b300.inputs import (WORKLOADS, Workload, gamma_schedule,
                                                            make_decode_inputs, make_grad_inputs,
                                                            make_inputs, theta_schedule, to_f64)
from oracle import retention_ref as O

from helpers import BF16_TOL, FP32_TOL, assert_close, gpu_np, head_slice, max_rel_inf, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_recurrent_sequence_prologue_b300 import build
    build.build()
    R.load()
    R.force_path(0)
    yield
    R.force_path(0)


def _cuda(inp):
    d = dict(inp)
    for key in ("q", "k", "v", "state_in"):
        if d.get(key) is not None:
            d[key] = d[key].cuda()
    return d


def _oracle_full(inp, w, form="chunkwise", chunk=None, pos0=0, gn=None):
    return O.retention(to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]),
                       np.asarray(inp["gamma"], np.float64), np.asarray(inp["theta"], np.float64),
                       pos0, to_f64(inp["state_in"]), form, chunk, gn)


def _custom(B, H, L, d_k, d_v, dtype, chunk, std=1.0, state_std=0.0, seed=0):
    assert dtype in ("f32", "bf16"), dtype
    w = Workload("custom", B, H, L, d_k, d_v, dtype, chunk, std, state_std=state_std)
    return w, make_inputs(w, seed)


# ---------------------------------------------------------------- prologue --
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_rotate_matches_oracle(dtype):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(2, 3, 200, 64, generator=g).to(dtype)
    th = theta_schedule(64)
    for pos0, scale in ((0, 1.0), (12345, 0.125)):
        y = R.rotate(x.cuda(), th, pos0=pos0, scale=scale, out_dtype=torch.float32)
        sin, cos = O.rotation_tables(np.arange(200) + pos0, th.astype(np.float64))
        ref = scale * O.theta_shift(to_f64(x), sin, cos)
        assert max_rel_inf(gpu_np(y), ref) < 2e-6


# ------------------------------------------------------------ fp32 (Tiny) --
def test_tiny_all_forms_vs_brute_force():
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, seed=0)
    ref_o, ref_s = O.brute_force(to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]),
                                 inp["gamma"].astype(np.float64), inp["theta"].astype(np.float64))
    d = _cuda(inp)
    o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk)
    assert_close(gpu_np(o), ref_o, torch.float32, "chunkwise")
    assert_close(gpu_np(s), ref_s, torch.float32, "chunkwise state")
    o2, s2 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk, layout="scan")
    assert torch.equal(s, s2) and torch.equal(o, o2)
    o3, s3 = R.parallel(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], return_state=True)
    assert_close(gpu_np(o3), ref_o, torch.float32, "parallel")
    assert_close(gpu_np(s3), ref_s, torch.float32, "parallel state")
    # recurrent form = 64 decode steps
    st = torch.zeros(1, 2, 16, 16, device="cuda")
    outs = [R.step(d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
                   d["v"][:, :, t].contiguous(), inp["gamma"], inp["theta"], t, st)
            for t in range(w.L)]
    assert_close(gpu_np(torch.stack(outs, 2)), ref_o, torch.float32, "steps")
    assert_close(gpu_np(st), ref_s, torch.float32, "steps state")


@pytest.mark.parametrize("L,chunk,pos0", [(64, 16, 0), (61, 16, 7), (50, 1, 3), (33, 64, 1000), (1, 16, 5)])
def test_fp32_edge_cases(L, chunk, pos0):
    w, inp = _custom(2, 3, L, 16, 12, "f32", chunk, state_std=0.3, seed=L)
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", chunk, pos0)
    d = _cuda(inp)
    o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=chunk, pos0=pos0,
                       state_in=d["state_in"])
    assert_close(gpu_np(o), ref_o, torch.float32, "out")
    assert_close(gpu_np(s), ref_s, torch.float32, "state")
    o2, s2 = R.parallel(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], pos0=pos0,
                        state_in=d["state_in"], return_state=True)
    assert_close(gpu_np(o2), ref_o, torch.float32, "parallel out")
    assert_close(gpu_np(s2), ref_s, torch.float32, "parallel state")


def test_groupnorm_fp32_with_affine():
    w, inp = _custom(2, 3, 48, 16, 24, "f32", 16, seed=9)
    gw = torch.randn(3 * 24, generator=torch.Generator().manual_seed(1))
    gbias = torch.randn(3 * 24, generator=torch.Generator().manual_seed(2))
    gn = {"eps": 1e-5, "weight": gw.reshape(3, 24).numpy(), "bias": gbias.reshape(3, 24).numpy()}
    ref_o, _ = _oracle_full(inp, w, "chunkwise", 16, 0, gn)
    d = _cuda(inp)
    o, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=16,
                       gn={"eps": 1e-5, "weight": gw.cuda(), "bias": gbias.cuda()})
    assert_close(gpu_np(o), ref_o, torch.float32, "gn")


@pytest.mark.parametrize("B,H,L,d_k,d_v,dtype,chunk,layout,out_f32,affine,pos0", [
    (1, 2, 300, 256, 256, "bf16", 128, "carry", False, True, 3),    # CTA pairs, short last chunk
    (2, 2, 300, 128, 128, "bf16", 128, "carry", True, False, 0),    # one-CTA kernel, fp32 out
    (1, 2, 1024, 256, 256, "bf16", 128, "scan", False, True, 5),    # chunk-parallel layout
    (3, 2, 200, 64, 64, "bf16", 64, "carry", False, True, [0, 37, 900]),   # per-row positions
    (1, 2, 130, 32, 20, "f32", 32, "carry", True, True, 0),         # fp32 path, 20-wide rows
])
def test_groupnorm_in_place_on_every_path(B, H, L, d_k, d_v, dtype, chunk, layout, out_f32, affine, pos0):
    """GroupNorm runs in place over the output after everything that writes
    it (the short-last-chunk copy included) on every path and layout."""
    w, inp = _custom(B, H, L, d_k, d_v, dtype, chunk, std=1.0, state_std=0.1, seed=L + d_v)
    g = torch.Generator().manual_seed(L)
    gw, gb = (torch.randn(H, d_v, generator=g) if affine else None for _ in range(2))
    d = _cuda(inp)
    gn = {"eps": 1e-5, "weight": gw.cuda() if affine else None, "bias": gb.cuda() if affine else None}
    o, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=chunk, pos0=pos0,
                       state_in=d["state_in"], gn=gn, layout=layout,
                       out_dtype=torch.float32 if out_f32 else None)
    assert R.sync_status() == R.RET_OK
    gref = {"eps": 1e-5, "weight": gw.numpy() if affine else None, "bias": gb.numpy() if affine else None}
    rows = pos0 if isinstance(pos0, list) else [pos0] * B
    tol = torch.float32 if dtype == "f32" else torch.bfloat16
    for b, p0 in enumerate(rows):
        one = {k: (v[b:b + 1] if torch.is_tensor(v) else v) for k, v in inp.items()}
        ref_o, _ = _oracle_full(one, w, "chunkwise", chunk, pos0=p0, gn=gref)
        assert_close(gpu_np(o[b:b + 1]), ref_o, tol, f"row {b}")


# ------------------------------------------------------- bf16, small shapes --
def test_small_workload_all_heads():
    w = WORKLOADS["small"]
    inp = make_inputs(w, seed=0)
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", w.chunk)
    d = _cuda(inp)
    o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk)
    assert R.sync_status() == R.RET_OK
    assert_close(gpu_np(o), ref_o, torch.bfloat16, "small out")
    assert_close(gpu_np(s), ref_s, torch.bfloat16, "small state")


@pytest.mark.parametrize("d_k,d_v,L,H", [(64, 128, 128, 1), (128, 128, 384, 2), (256, 256, 512, 2),
                                         (256, 512, 256, 3)])
def test_tc_chunkwise_vs_oracle(d_k, d_v, L, H):
    w, inp = _custom(2, H, L, d_k, d_v, "bf16", 128, std=1.0, state_std=0.1, seed=d_k + L)
    path, _ = R.plan("chunkwise", torch.bfloat16, 2, H, L, d_k, d_v, 128, gamma=inp["gamma"])
    assert path == R.RET_PATH_TC
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", 128, pos0=17)
    d = _cuda(inp)
    for odt in (torch.bfloat16, torch.float32):
        o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=17,
                           state_in=d["state_in"], out_dtype=odt)
        assert R.sync_status() == R.RET_OK
        assert_close(gpu_np(o), ref_o, torch.bfloat16, f"tc out {odt}")
        assert_close(gpu_np(s), ref_s, torch.bfloat16, "tc state")


def test_tc_matches_fp32_kernels():
    w, inp = _custom(1, 2, 256, 256, 256, "bf16", 128, state_std=0.1, seed=5)
    d = _cuda(inp)
    o_tc, s_tc = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128,
                             state_in=d["state_in"], out_dtype=torch.float32)
    R.force_path(R.RET_PATH_SIMT)
    try:
        o_f, s_f = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128,
                               state_in=d["state_in"], out_dtype=torch.float32)
    finally:
        R.force_path(0)
    assert_close(gpu_np(o_tc), gpu_np(o_f), torch.bfloat16, "tensor cores vs fp32 kernels, out")
    assert_close(gpu_np(s_tc), gpu_np(s_f), torch.bfloat16, "tensor cores vs fp32 kernels, state")


@pytest.mark.parametrize("path", [0, 2])
def test_exact_causality_on_gpu(path):
    """Outputs before position m are bit-identical when inputs at ≥ m change."""
    w, inp = _custom(1, 2, 384, 128, 128, "bf16", 128, state_std=0.1, seed=11)
    d = _cuda(inp)
    m = 200
    q2, k2, v2 = d["q"].clone(), d["k"].clone(), d["v"].clone()
    gen = torch.Generator(device="cuda").manual_seed(4)
    for t in (q2, k2, v2):
        t[:, :, m:] = (torch.randn(t[:, :, m:].shape, generator=gen, device="cuda") * 3).to(t.dtype)
    R.force_path(path)
    try:
        o1, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, state_in=d["state_in"])
        o2, _ = R.chunkwise(q2, k2, v2, inp["gamma"], inp["theta"], chunk=128, state_in=d["state_in"])
    finally:
        R.force_path(0)
    assert torch.equal(o1[:, :, :m], o2[:, :, :m])
    assert not torch.equal(o1[:, :, m:], o2[:, :, m:])


def test_split_call_consistency_tc():
    w, inp = _custom(1, 2, 512, 256, 128, "bf16", 128, state_std=0.1, seed=12)
    d = _cuda(inp)
    o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=5,
                       state_in=d["state_in"], out_dtype=torch.float32)
    h = 256
    sl = lambda t, a, b: t[:, :, a:b].contiguous()
    oa, sa = R.chunkwise(sl(d["q"], 0, h), sl(d["k"], 0, h), sl(d["v"], 0, h), inp["gamma"],
                         inp["theta"], chunk=128, pos0=5, state_in=d["state_in"], out_dtype=torch.float32)
    ob, sb = R.chunkwise(sl(d["q"], h, 512), sl(d["k"], h, 512), sl(d["v"], h, 512), inp["gamma"],
                         inp["theta"], chunk=128, pos0=5 + h, state_in=sa, out_dtype=torch.float32)
    assert torch.equal(torch.cat([oa, ob], 2), o)
    assert torch.equal(sb, s)


@pytest.mark.parametrize("d_k,d_v,L,H", [(64, 128, 384, 2), (256, 512, 512, 2)])
def test_tc_scan_layout_is_bit_identical_to_carry(d_k, d_v, L, H):
    """Chunk-parallel layout (ΔS per chunk, fp32 scan, outputs from entering
    states) against the carried-state layout: same state and outputs, bit for bit."""
    w, inp = _custom(2, H, L, d_k, d_v, "bf16", 128, std=1.0, state_std=0.1, seed=d_k + 7)
    path, _ = R.plan("chunkwise_scan", torch.bfloat16, 2, H, L, d_k, d_v, 128, gamma=inp["gamma"])
    assert path == R.RET_PATH_TC
    d = _cuda(inp)
    for odt in (torch.bfloat16, torch.float32):
        R.force_path(R.RET_PATH_TC_CARRY)   # keep the carried layout for a grid this small
        try:
            o1, s1 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=9,
                                 state_in=d["state_in"], out_dtype=odt)
        finally:
            R.force_path(0)
        o2, s2 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=9,
                             state_in=d["state_in"], out_dtype=odt, layout="scan")
        assert R.sync_status() == R.RET_OK
        assert torch.equal(s1, s2)
        assert torch.equal(o1, o2)
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", 128, pos0=9)
    assert_close(gpu_np(o2), ref_o, torch.bfloat16, "scan out")
    assert_close(gpu_np(s2), ref_s, torch.bfloat16, "scan state")


@pytest.mark.parametrize("d_k,L,H,chunk,pos0", [(64, 640, 3, 64, 0), (128, 300, 2, 128, 9), (256, 129, 1, 64, 40)])
def test_tc_narrow_value_tile(d_k, L, H, chunk, pos0):
    """d_v = 64 on the tensor cores (the Small MSR shape): one 128-wide tile of
    which the first 64 columns are live; a requested chunk of 64 runs on the
    128-token tile.  Carried and chunk-parallel layouts give the same bits;
    against the oracle at the requested chunk."""
    w, inp = _custom(2, H, L, d_k, 64, "bf16", chunk, std=0.125, state_std=0.1, seed=L + d_k)
    path, _ = R.plan("chunkwise", torch.bfloat16, 2, H, L, d_k, 64, chunk, gamma=inp["gamma"])
    assert path == R.RET_PATH_TC
    d = _cuda(inp)
    res = {}
    for layout in ("carry", "scan"):
        R.force_path(R.RET_PATH_TC_CARRY if layout == "carry" else 0)
        try:
            for odt in (torch.bfloat16, torch.float32):
                res[layout, odt] = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"],
                                               chunk=chunk, pos0=pos0, state_in=d["state_in"],
                                               out_dtype=odt, layout=layout)
                assert R.sync_status() == R.RET_OK
        finally:
            R.force_path(0)
    for odt in (torch.bfloat16, torch.float32):
        assert torch.equal(res["carry", odt][0], res["scan", odt][0])
        assert torch.equal(res["carry", odt][1], res["scan", odt][1])
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", chunk, pos0=pos0)
    o, s = res["carry", torch.float32]
    assert_close(gpu_np(o), ref_o, torch.bfloat16, "d_v 64 out")
    assert_close(gpu_np(s), ref_s, torch.bfloat16, "d_v 64 state")
    # the idle columns write nothing: out and state_out are views at the start
    # of NaN-filled buffers whose tails must stay NaN, and the values match
    n, m = 2 * H * L * 64, 2 * H * d_k * 64
    ob = torch.full((n + 128 * 128,), float("nan"), dtype=torch.bfloat16, device="cuda")
    sb = torch.full((m + 128 * 128,), float("nan"), dtype=torch.float32, device="cuda")
    for layout in ("carry", "scan"):
        R.force_path(R.RET_PATH_TC_CARRY if layout == "carry" else 0)
        try:
            o2, s2 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=chunk, pos0=pos0,
                                 state_in=d["state_in"], out=ob[:n].view(2, H, L, 64),
                                 state_out=sb[:m].view(2, H, d_k, 64), layout=layout)
            assert R.sync_status() == R.RET_OK
        finally:
            R.force_path(0)
        assert torch.equal(o2, res["carry", torch.bfloat16][0]) and torch.equal(s2, res["carry", torch.bfloat16][1])
        assert torch.isnan(ob[n:].float()).all() and torch.isnan(sb[m:]).all()


@pytest.mark.parametrize("d_k,d_v,L,H", [(256, 256, 512, 2), (128, 512, 384, 1), (256, 512, 640, 2)])
def test_tc_pair_kernel_matches_single_cta_kernel(d_k, d_v, L, H):
    """The CTA-pair chunk kernel (cta_group::2, two d_v tiles per cluster)
    against the one-CTA-per-tile kernel: the same products in the same
    order, so the same bits, for outputs and state, on every layout."""
    w, inp = _custom(2, H, L, d_k, d_v, "bf16", 128, std=1.0, state_std=0.1, seed=d_k + 3 * L)
    d = _cuda(inp)
    res = {}
    try:
        for mode in (0, R.RET_PATH_TC_SINGLE):
            R.force_path(mode)
            for odt in (torch.bfloat16, torch.float32):
                for layout in ("carry", "scan"):
                    res[mode, odt, layout] = R.chunkwise(
                        d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=11,
                        state_in=d["state_in"], out_dtype=odt, layout=layout)
                    assert R.sync_status() == R.RET_OK
    finally:
        R.force_path(0)
    for key, (o, s) in res.items():
        o1, s1 = res[R.RET_PATH_TC_SINGLE, key[1], key[2]]
        assert torch.equal(s, s1), key
        assert torch.equal(o, o1), key
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", 128, pos0=11)
    o, s = res[0, torch.float32, "carry"]
    assert_close(gpu_np(o), ref_o, torch.bfloat16, "pair out")
    assert_close(gpu_np(s), ref_s, torch.bfloat16, "pair state")


@pytest.mark.parametrize("B,H,L,d_k,d_v,rowpos", [
    (2, 2, 1024, 256, 512, False),   # 8 chunks: every ring slot used twice
    (1, 3, 1300, 256, 256, False),   # 11 chunks, the last of 20 tokens
    (2, 40, 260, 256, 512, False),   # 80 heads: three launches of 32, 32 and 16 heads
    (3, 2, 700, 128, 256, True),     # d_k 128, one start position per batch row
    (1, 2, 900, 256, 256, False),    # 8 chunks, the last of 4 tokens
])
def test_compact_workspace_matches_front_pass(B, H, L, d_k, d_v, rowpos):
    """The compact-workspace mode of the carried layout on CTA pairs (the Θ
    prologue fused into the launch: producer CTAs rotating q, k into an
    L2-resident ring of chunk slots) against the same kernels fed by the
    front pass over the whole sequence, and against the chunk-parallel
    layout: the same Q″ and K̂′ bits reach the same products, so out and
    state agree bit for bit."""
    w, inp = _custom(B, H, L, d_k, d_v, "bf16", 128, std=1.0, state_std=0.1, seed=L + H)
    d = _cuda(inp)
    pos = [0, 37, 5000][:B] if rowpos else 13
    full = R.plan("chunkwise", torch.bfloat16, B, H, L, d_k, d_v, 128)[1]
    small = R.plan("chunkwise_compact", torch.bfloat16, B, H, L, d_k, d_v, 128)[1]
    assert small < full
    res = {}
    for compact in (True, False):
        for odt in (torch.bfloat16, torch.float32):
            res[compact, odt] = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"],
                                            chunk=128, pos0=pos, state_in=d["state_in"], out_dtype=odt,
                                            compact=compact)
            assert R.sync_status() == R.RET_OK
    for odt in (torch.bfloat16, torch.float32):
        o, s = res[True, odt]
        o1, s1 = res[False, odt]
        assert torch.equal(s, s1), odt
        assert torch.equal(o, o1), odt
        if not rowpos:
            o2, s2 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128,
                                 pos0=pos, state_in=d["state_in"], out_dtype=odt, layout="scan")
            assert torch.equal(s, s2) and torch.equal(o, o2), odt
    o, s = res[True, torch.float32]
    for b in range(B):
        for h in (0, H - 1):
            one = {k: (v[b:b + 1, h:h + 1] if torch.is_tensor(v) else v) for k, v in inp.items()}
            one["gamma"] = inp["gamma"][h:h + 1]
            ref_o, ref_s = _oracle_full(one, w, "chunkwise", 128, pos0=pos[b] if rowpos else pos)
            assert_close(gpu_np(o[b:b + 1, h:h + 1]), ref_o, torch.bfloat16, f"ring out (b={b},h={h})")
            assert_close(gpu_np(s[b:b + 1, h:h + 1]), ref_s, torch.bfloat16, f"ring state (b={b},h={h})")


@pytest.mark.parametrize("d_k,d_v,L,H", [
    (256, 512, 300, 2),    # pair kernel, short last chunk of 44
    (256, 256, 1000, 1),   # pair kernel, 8 chunks, last of 104
    (256, 256, 77, 2),     # pair kernel, one short chunk
    (128, 128, 200, 2),    # one-CTA kernel
    (64, 128, 129, 2),     # one-CTA kernel, last chunk of 1 token
    (256, 256, 1, 2),      # pair kernel, a single token
    (128, 128, 1, 3),      # one-CTA kernel, a single token
])
def test_tc_ragged_length_vs_oracle(d_k, d_v, L, H):
    """L not a multiple of the chunk on the tensor-core path: the rotated
    workspace is padded with zero rows, V is read per head (zeros past L),
    the last chunk carries with γ^{L mod 128} and its outputs stop at L.
    Against the oracle; carry and chunk-parallel layouts agree bit for bit,
    and so do the pair and one-CTA kernels."""
    w, inp = _custom(2, H, L, d_k, d_v, "bf16", 128, std=1.0, state_std=0.1, seed=L + d_k)
    path, _ = R.plan("chunkwise", torch.bfloat16, 2, H, L, d_k, d_v, 128, gamma=inp["gamma"])
    assert path == R.RET_PATH_TC
    d = _cuda(inp)
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", 128, pos0=21)
    res = {}
    try:
        for mode in (0, R.RET_PATH_TC_SINGLE):
            R.force_path(mode)
            for odt in (torch.bfloat16, torch.float32):
                for layout in ("carry", "scan"):
                    res[mode, odt, layout] = R.chunkwise(
                        d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=21,
                        state_in=d["state_in"], out_dtype=odt, layout=layout)
                    assert R.sync_status() == R.RET_OK
    finally:
        R.force_path(0)
    for (mode, odt, layout), (o, s) in res.items():
        o0, s0 = res[0, odt, "carry"]
        assert torch.equal(s, s0), (mode, odt, layout)
        assert torch.equal(o, o0), (mode, odt, layout)
    o, s = res[0, torch.float32, "carry"]
    assert_close(gpu_np(o), ref_o, torch.bfloat16, "ragged out")
    assert_close(gpu_np(s), ref_s, torch.bfloat16, "ragged state")
    # nothing is written past row L of any head: the output is a view at the
    # start of a NaN-filled buffer whose tail (a chunk's worth of rows) must stay NaN
    n = 2 * H * L * d_v
    big = torch.full((n + 128 * d_v,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o2, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=21,
                        state_in=d["state_in"], out=big[:n].view(2, H, L, d_v))
    assert R.sync_status() == R.RET_OK
    assert torch.equal(o2, res[0, torch.bfloat16, "carry"][0])
    assert torch.isnan(big[n:].float()).all()


@pytest.mark.parametrize("dtype,d_k,d_v,L,H", [
    ("bf16", 256, 256, 300, 2),   # tensor cores (CTA pairs, short last chunk)
    ("bf16", 128, 128, 256, 1),   # tensor cores (one CTA per tile)
    ("f32", 32, 24, 96, 2),       # fp32 path
])
def test_rowpos_vs_oracle(dtype, d_k, d_v, L, H):
    """ret_chunkwise_rowpos: each batch row at its own start position, against
    the oracle run row by row; with one shared start it equals ret_chunkwise
    bit for bit."""
    B = 3
    w, inp = _custom(B, H, L, d_k, d_v, dtype, 128 if dtype == "bf16" else 32, std=1.0,
                     state_std=0.1, seed=L + H)
    d = _cuda(inp)
    rows = [0, 37, 5000]
    o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk, pos0=rows,
                       state_in=d["state_in"], out_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    for b, p0 in enumerate(rows):
        one = {k: (v[b:b + 1] if torch.is_tensor(v) else v) for k, v in inp.items()}
        ref_o, ref_s = _oracle_full(one, w, "chunkwise", w.chunk, pos0=p0)
        assert_close(gpu_np(o[b:b + 1]), ref_o, w.torch_dtype, f"row {b} out")
        assert_close(gpu_np(s[b:b + 1]), ref_s, w.torch_dtype, f"row {b} state")
    o1, s1 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk,
                         pos0=[41] * B, state_in=d["state_in"])
    o2, s2 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk, pos0=41,
                         state_in=d["state_in"])
    assert R.sync_status() == R.RET_OK
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("d_k,d_v,L,H,state", [(64, 128, 256, 1, False), (128, 256, 384, 2, True),
                                               (256, 512, 512, 2, True)])
def test_tc_parallel_form_vs_oracle(d_k, d_v, L, H, state):
    """ret_parallel on the tensor cores: block-tiled (Q′K′ᵀ ⊙ D)V, no recurrence."""
    w, inp = _custom(2, H, L, d_k, d_v, "bf16", 128, std=1.0, state_std=0.1 if state else 0.0,
                     seed=d_k + L)
    path, _ = R.plan("parallel", torch.bfloat16, 2, H, L, d_k, d_v, gamma=inp["gamma"],
                     state_out=True)
    assert path == R.RET_PATH_TC
    ref_o, ref_s = _oracle_full(inp, w, "parallel", pos0=5)
    d = _cuda(inp)
    for odt in (torch.bfloat16, torch.float32):
        o, s = R.parallel(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], pos0=5,
                          state_in=d["state_in"], return_state=True, out_dtype=odt)
        assert R.sync_status() == R.RET_OK
        assert_close(gpu_np(o), ref_o, torch.bfloat16, f"parallel out {odt}")
        assert_close(gpu_np(s), ref_s, torch.bfloat16, "parallel state")
    # the parallel and chunkwise forms agree closely; the final state is the same bits
    oc, sc = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=128, pos0=5,
                         state_in=d["state_in"], out_dtype=torch.float32)
    assert rel_fro(gpu_np(o), gpu_np(oc)) < 1e-2
    assert torch.equal(s, sc)


def test_tc_parallel_groupnorm_and_causality():
    w, inp = _custom(1, 2, 384, 128, 128, "bf16", 128, std=1.0, seed=31)
    gn = {"eps": 1e-5}
    ref_o, _ = _oracle_full(inp, w, "parallel", gn=gn)
    d = _cuda(inp)
    o, _ = R.parallel(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], gn=gn)
    assert_close(gpu_np(o), ref_o, torch.bfloat16, "parallel gn")
    m = 200
    q2, k2, v2 = d["q"].clone(), d["k"].clone(), d["v"].clone()
    for t in (q2, k2, v2):
        t[:, :, m:] = 3.0
    o1, _ = R.parallel(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"])
    o2, _ = R.parallel(q2, k2, v2, inp["gamma"], inp["theta"])
    assert torch.equal(o1[:, :, :m], o2[:, :, :m])


# -------------------------------------------------------- full workloads --
def test_msr1p3b_groupnorm_all_heads():
    """The 1.3B-shape workload (GroupNorm on) against the oracle on all 64 (b, h)."""
    w = WORKLOADS["msr1p3b"]
    inp = make_inputs(w, seed=0)
    d = _cuda(inp)
    o, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk,
                       gn={"eps": w.gn_eps}, return_state=False)
    assert R.sync_status() == R.RET_OK
    og = gpu_np(o)
    for b in range(w.B):
        for h in range(w.H):
            q, k, v, s, g, th = head_slice(inp, b, h)
            ref, _ = O.retention(q, k, v, g, th, 0, s, "chunkwise", w.chunk, {"eps": w.gn_eps})
            assert_close(og[b:b + 1, h:h + 1], ref, torch.bfloat16, f"1.3B (b={b},h={h})")


def test_msr7b_all_heads():
    """The 7B-shape workload against the oracle on all 32 (b, h), out and state."""
    w = WORKLOADS["msr7b"]
    inp = make_inputs(w, seed=0)
    d = _cuda(inp)
    o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk,
                       state_in=d["state_in"])
    assert R.sync_status() == R.RET_OK
    # full size: the chunk-parallel layout returns the same bits
    o2, s2 = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk,
                         state_in=d["state_in"], layout="scan")
    assert R.sync_status() == R.RET_OK
    assert torch.equal(s, s2) and torch.equal(o, o2)
    del o2, s2
    og, sg = gpu_np(o), gpu_np(s)
    for b in range(w.B):
        for h in range(w.H):
            q, k, v, si, g, th = head_slice(inp, b, h)
            ref_o, ref_s = O.retention(q, k, v, g, th, 0, si, "chunkwise", w.chunk)
            assert_close(og[b:b + 1, h:h + 1], ref_o, torch.bfloat16, f"7B out (b={b},h={h})")
            assert_close(sg[b:b + 1, h:h + 1], ref_s, torch.bfloat16, f"7B state (b={b},h={h})")


# --------------------------------------------------------------- gradients --
def _oracle_bwd(inp, gi, pos0):
    return O.retention_backward(to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]),
                                np.asarray(inp["gamma"], np.float64),
                                np.asarray(inp["theta"], np.float64), pos0,
                                to_f64(inp["state_in"]), to_f64(gi["d_out"]),
                                to_f64(gi["d_state_out"]))


@pytest.mark.parametrize("dtype,gdtype,B,H,L,d_k,d_v,chunk,pos0,state,dso", [
    # fp32 kernels
    ("f32", torch.float32, 2, 3, 300, 64, 96, 64, 7, True, True),       # 5 chunks, ragged
    ("f32", torch.float32, 1, 2, 77, 32, 768, 100, 0, True, False),     # one chunk, wide d_v
    ("f32", torch.bfloat16, 1, 1, 65, 2, 1, 16, 40, False, False),      # smallest widths
    ("bf16", torch.bfloat16, 1, 2, 200, 256, 256, 48, 3, True, True),   # chunk 48
    # tensor cores
    ("bf16", torch.float32, 2, 2, 256, 128, 128, 128, 100, False, True),   # one-CTA kernels
    ("bf16", torch.float32, 1, 2, 300, 256, 512, 128, 5, True, True),      # two d_v pieces, pairs, ragged
    ("bf16", torch.bfloat16, 1, 3, 200, 128, 384, 128, 0, True, True),     # pieces of 256 and 128
    ("bf16", torch.float32, 2, 2, 1, 256, 256, 128, 9, True, True),        # a single token
    ("bf16", torch.float32, 1, 2, 260, 128, 256, 128, 2, True, True),      # dV on d_k = 128 CTA pairs
    ("bf16", torch.bfloat16, 1, 2, 140, 256, 384, 128, 6, True, True),     # a 128-wide piece on d_k = 128 pairs
])
def test_backward_vs_oracle(dtype, gdtype, B, H, L, d_k, d_v, chunk, pos0, state, dso):
    w, inp = _custom(B, H, L, d_k, d_v, dtype, chunk, state_std=0.1 if state else 0.0)
    gi = make_grad_inputs(w, seed=5, d_state_std=1.0 if dso else 0.0)
    ref = _oracle_bwd(inp, gi, pos0)
    path, _ = R.backward_plan(w.torch_dtype, B, H, L, d_k, d_v, chunk, gamma=inp["gamma"])
    assert path == (R.RET_PATH_TC if dtype == "bf16" and chunk == 128 else R.RET_PATH_SIMT)
    d = _cuda(inp)
    dso_c = gi["d_state_out"].cuda() if dso else None
    got = R.chunkwise_backward(d["q"], d["k"], d["v"], gi["d_out"].cuda(), inp["gamma"], inp["theta"],
                               chunk=chunk, pos0=pos0, state_in=d["state_in"], d_state_out=dso_c,
                               grad_dtype=gdtype)
    assert R.sync_status() == R.RET_OK
    for g, r, name in zip(got, ref, ("dq", "dk", "dv", "dS_in")):
        # fp32 kernels: fp32 tolerance unless the gradients are stored in bf16;
        # tensor cores: bf16 operands, the bf16 tolerance
        tol = torch.bfloat16 if (path == R.RET_PATH_TC or (gdtype == torch.bfloat16 and name != "dS_in")) \
            else torch.float32
        assert_close(gpu_np(g), r, tol, name)


@pytest.mark.parametrize("dtype,d,chunk", [("f32", 64, 32), ("bf16", 128, 128)])
def test_backward_zero_upstream_and_state_aliasing(dtype, d, chunk):
    w, inp = _custom(1, 2, 130, d, d, dtype, chunk, state_std=0.1)
    d_ = _cuda(inp)
    # zero upstream gradients give exactly zero gradients
    z = torch.zeros((1, 2, 130, d), device="cuda", dtype=w.torch_dtype)
    zs = torch.zeros((1, 2, d, d), device="cuda")
    got = R.chunkwise_backward(d_["q"], d_["k"], d_["v"], z, inp["gamma"], inp["theta"], chunk=chunk,
                               state_in=d_["state_in"], d_state_out=zs)
    assert all(int(torch.count_nonzero(t)) == 0 for t in got)
    # d_state_in written over d_state_out: the same values as into a separate buffer
    gi = make_grad_inputs(w, seed=2, d_state_std=1.0)
    dso = gi["d_state_out"].cuda()
    a = R.chunkwise_backward(d_["q"], d_["k"], d_["v"], gi["d_out"].cuda(), inp["gamma"],
                             inp["theta"], chunk=chunk, pos0=9, state_in=d_["state_in"], d_state_out=dso)
    buf = dso.clone()
    b = R.chunkwise_backward(d_["q"], d_["k"], d_["v"], gi["d_out"].cuda(), inp["gamma"],
                             inp["theta"], chunk=chunk, pos0=9, state_in=d_["state_in"], d_state_out=buf,
                             d_state_in=buf)
    assert R.sync_status() == R.RET_OK
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("L", [130, 256])
def test_backward_tc_smallest_gamma(L):
    """The tensor-core gradient pass at the γ bound of its path (γ^255 just
    above 2^-100): the anti-causal evaluations start from γ^{r−256}·dS_out,
    about 2^96 · dS_out for the ragged length, and must still match the
    oracle."""
    w, inp = _custom(1, 2, L, 128, 128, "bf16", 128, state_std=0.1, seed=31)
    inp["gamma"] = np.array([0.77, 0.999], np.float32)
    gi = make_grad_inputs(w, seed=32, d_state_std=1.0)
    path, _ = R.backward_plan(w.torch_dtype, 1, 2, L, 128, 128, 128, gamma=inp["gamma"])
    assert path == R.RET_PATH_TC
    ref = _oracle_bwd(inp, gi, 3)
    d = _cuda(inp)
    got = R.chunkwise_backward(d["q"], d["k"], d["v"], gi["d_out"].cuda(), inp["gamma"], inp["theta"],
                               chunk=128, pos0=3, state_in=d["state_in"],
                               d_state_out=gi["d_state_out"].cuda(), grad_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    for g, r, name in zip(got, ref, ("dq", "dk", "dv", "dS_in")):
        assert np.isfinite(gpu_np(g)).all(), name
        assert_close(gpu_np(g), r, torch.bfloat16, name)


def test_backward_tc_matches_fp32_kernels():
    """The tensor-core gradient pass against the fp32 kernels on the same bf16 inputs."""
    w, inp = _custom(2, 2, 384, 256, 256, "bf16", 128, state_std=0.1, seed=21)
    gi = make_grad_inputs(w, seed=22, d_state_std=1.0)
    d = _cuda(inp)
    args = (d["q"], d["k"], d["v"], gi["d_out"].cuda(), inp["gamma"], inp["theta"])
    kw = dict(chunk=128, pos0=17, state_in=d["state_in"], d_state_out=gi["d_state_out"].cuda(),
              grad_dtype=torch.float32)
    tc = R.chunkwise_backward(*args, **kw)
    R.force_path(R.RET_PATH_SIMT)
    try:
        ref = R.chunkwise_backward(*args, **kw)
    finally:
        R.force_path(0)
    assert R.sync_status() == R.RET_OK
    for x, y, name in zip(tc, ref, ("dq", "dk", "dv", "dS_in")):
        assert_close(gpu_np(x), gpu_np(y), torch.bfloat16, name)


def test_backward_msr7b_sampled_heads():
    """The 7B shape (bf16 inputs, fp32 gradients, tensor-core path): one head
    against the oracle over the whole sequence; another on the prefix that
    fixes dq (positions ≤ t and S_in) and the suffix that fixes dk, dv
    (positions ≥ m and dS_out)."""
    w = WORKLOADS["msr7b"]
    inp = make_inputs(w, seed=0)
    gi = make_grad_inputs(w, seed=5, d_state_std=1.0)
    d = _cuda(inp)
    dq, dk, dv, dsi = R.chunkwise_backward(d["q"], d["k"], d["v"], gi["d_out"].cuda(), inp["gamma"],
                                           inp["theta"], chunk=w.chunk, state_in=d["state_in"],
                                           d_state_out=gi["d_state_out"].cuda(),
                                           grad_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    b, h = 1, 15
    q, k, v, si, g, th = head_slice(inp, b, h)
    dO = to_f64(gi["d_out"][b:b + 1, h:h + 1])
    dSo = to_f64(gi["d_state_out"][b:b + 1, h:h + 1])
    ref = O.retention_backward(q, k, v, g, th, 0, si, dO, dSo)
    for got, r, name in zip((dq, dk, dv, dsi), ref, ("dq", "dk", "dv", "dS_in")):
        assert_close(gpu_np(got[b:b + 1, h:h + 1]), r, torch.bfloat16, f"7B {name} (b={b},h={h})")
    b, h, n = 0, 0, 384
    q, k, v, si, g, th = head_slice(inp, b, h)
    dO = to_f64(gi["d_out"][b:b + 1, h:h + 1])
    dSo = to_f64(gi["d_state_out"][b:b + 1, h:h + 1])
    rq = O.retention_backward(q[:, :, :n], k[:, :, :n], v[:, :, :n], g, th, 0, si, dO[:, :, :n])[0]
    assert_close(gpu_np(dq[b:b + 1, h:h + 1, :n]), rq, torch.bfloat16, "7B dq prefix")
    m0 = w.L - n
    _, rk, rv, _ = O.retention_backward(q[:, :, m0:], k[:, :, m0:], v[:, :, m0:], g, th, m0, None,
                                        dO[:, :, m0:], dSo)
    assert_close(gpu_np(dk[b:b + 1, h:h + 1, m0:]), rk, torch.bfloat16, "7B dk suffix")
    assert_close(gpu_np(dv[b:b + 1, h:h + 1, m0:]), rv, torch.bfloat16, "7B dv suffix")


# ------------------------------------------------- row-normalised decay --
@pytest.mark.parametrize("dtype,d_k,d_v,L,chunk,pos0,state", [
    ("bf16", 256, 256, 300, 128, 0, True),     # tensor-core output, ragged
    ("bf16", 128, 128, 256, 128, 7, False),
    ("f32", 16, 24, 70, 16, 500, True),        # fp32 kernels
    ("bf16", 32, 36, 100, 32, 3, True),        # rows of 72 bytes: the element-wise pass
])
def test_decay_row_norm_vs_oracle(dtype, d_k, d_v, L, chunk, pos0, state):
    w, inp = _custom(2, 3, L, d_k, d_v, dtype, chunk, state_std=0.1 if state else 0.0, seed=L + pos0)
    d = _cuda(inp)
    o, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=chunk, pos0=pos0,
                       state_in=d["state_in"], return_state=False)
    R.decay_row_norm(o, inp["gamma"], pos0=pos0)
    assert R.sync_status() == R.RET_OK
    ref = O.normalised_retention(to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]),
                                 np.asarray(inp["gamma"], np.float64),
                                 np.asarray(inp["theta"], np.float64), pos0, to_f64(inp["state_in"]))
    assert_close(gpu_np(o), ref, w.torch_dtype, "row-normalised")


def test_decay_row_norm_decode_step():
    """A decode step's output at position pos, normalised by r_pos."""
    g = torch.Generator().manual_seed(41)
    q, k = torch.randn(2, 4, 64, generator=g), torch.randn(2, 4, 64, generator=g)
    v, S = torch.randn(2, 4, 128, generator=g), 0.1 * torch.randn(2, 4, 64, 128, generator=g)
    gam, th = gamma_schedule(4), theta_schedule(64)
    st = S.cuda()
    out = R.step(q.cuda(), k.cuda(), v.cuda(), gam, th, 1234, st)
    R.decay_row_norm(out, gam, pos0=1234)
    ref = O.normalised_retention(to_f64(q)[:, :, None], to_f64(k)[:, :, None], to_f64(v)[:, :, None],
                                 gam.astype(np.float64), th.astype(np.float64), 1234, to_f64(S))
    assert_close(gpu_np(out)[:, :, None], ref, torch.float32, "decode row-normalised")


def test_decode_1024_steps_vs_chunkwise_and_oracle():
    w = WORKLOADS["decode"]
    inp = make_decode_inputs(w, seed=0, device="cuda")
    S0 = inp["state"]
    st = S0.clone()
    outs = torch.empty((w.steps, w.B, w.H, w.d_v), dtype=torch.bfloat16, device="cuda")
    for t in range(w.steps):
        R.step(inp["q"][t], inp["k"][t], inp["v"][t], inp["gamma"], inp["theta"], t, st, out=outs[t])
    assert R.sync_status() == R.RET_OK
    q = inp["q"].permute(1, 2, 0, 3).contiguous()
    k = inp["k"].permute(1, 2, 0, 3).contiguous()
    v = inp["v"].permute(1, 2, 0, 3).contiguous()
    oc, sc = R.chunkwise(q, k, v, inp["gamma"], inp["theta"], chunk=128, state_in=S0)
    od = outs.permute(1, 2, 0, 3)
    assert_close(gpu_np(od), gpu_np(oc), torch.bfloat16, "decode vs chunkwise, out")
    assert_close(gpu_np(st), gpu_np(sc), torch.bfloat16, "decode vs chunkwise, state")
    # 17 heads against the float64 recurrent form: the even heads of batch row
    # 0, the odd heads of row 127 (so the first and the last (b, h)) and one
    # in between
    heads = [(0, h) for h in range(w.H)[::2]] + [(127, h) for h in range(w.H)[1::2]] + [(77, 9)]
    for b, h in heads:
        ref_o, ref_s = O.retention(to_f64(q[b:b + 1, h:h + 1]), to_f64(k[b:b + 1, h:h + 1]),
                                   to_f64(v[b:b + 1, h:h + 1]), inp["gamma"][h:h + 1].astype(np.float64),
                                   inp["theta"].astype(np.float64), 0, to_f64(S0[b:b + 1, h:h + 1]),
                                   "recurrent")
        assert_close(gpu_np(od[b:b + 1, h:h + 1]), ref_o, torch.bfloat16, f"decode (b={b},h={h})")
        assert_close(gpu_np(st[b:b + 1, h:h + 1]), ref_s, torch.bfloat16, f"decode state (b={b},h={h})")


def test_decode_groupnorm_and_odd_width():
    w, inp = _custom(3, 2, 1, 32, 30, "bf16", 1, state_std=0.1, seed=21)
    d = _cuda(inp)
    st = d["state_in"].clone()
    o = R.step(d["q"][:, :, 0].contiguous(), d["k"][:, :, 0].contiguous(), d["v"][:, :, 0].contiguous(),
               inp["gamma"], inp["theta"], 41, st, out_dtype=torch.float32, gn={"eps": 1e-5})
    ref_o, ref_s = O.decode_step(to_f64(inp["q"][:, :, 0]), to_f64(inp["k"][:, :, 0]),
                                 to_f64(inp["v"][:, :, 0]), inp["gamma"].astype(np.float64),
                                 inp["theta"].astype(np.float64), 41, to_f64(inp["state_in"]),
                                 {"eps": 1e-5})
    assert_close(gpu_np(o), ref_o, torch.bfloat16, "decode gn")
    assert max_rel_inf(gpu_np(st), ref_s) < 1e-5


# -------------------------------------------------------- failure path --
def test_bounded_wait_timeout_reports_and_recovers():
    assert R.sync_status() == R.RET_OK
    R.selftest_timeout(2000)
    assert R.sync_status() == R.RET_ETIMEOUT
    assert R.sync_status() == R.RET_OK
    w, inp = _custom(1, 2, 64, 16, 16, "f32", 16, seed=1)
    d = _cuda(inp)
    o, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=16)
    ref_o, _ = _oracle_full(inp, w, "chunkwise", 16)
    assert_close(gpu_np(o), ref_o, torch.float32, "after timeout")


# ----------------------------------------------------- grids past 65535 rows --
def test_folded_grids_match_unfolded_launches():
    """Launches with more rows than one grid dimension holds fold them over
    two: the fp32 chunk kernels (B·H·⌈L/chunk⌉ > 65535, forward and
    gradient pass), the Θ rotation (more than 65535 groups of 8 rows) and
    the tensor-core chunk-parallel layout (B·H·⌈L/128⌉ > 65535 CTA rows).
    Each against the same problem in launches that fit one dimension: the
    chunkwise result does not depend on the chunk length (fp32: to rounding),
    and the chunk-parallel layout equals the carried one bit for bit."""
    g = torch.Generator().manual_seed(41)
    # fp32 path: 2 heads × 40000 chunks of 1 token
    q, k, v = (torch.randn(1, 2, 40000, 8, generator=g) for _ in range(3))
    s0 = torch.randn(1, 2, 8, 8, generator=g) * 0.1
    gam, th = np.array([0.9, 0.99], np.float32), theta_schedule(8)
    qc, kc, vc, sc = q.cuda(), k.cuda(), v.cuda(), s0.cuda()
    o1, s1 = R.chunkwise(qc, kc, vc, gam, th, chunk=1, pos0=5, state_in=sc)
    o2, s2 = R.chunkwise(qc, kc, vc, gam, th, chunk=64, pos0=5, state_in=sc)
    d_o = torch.randn(1, 2, 40000, 8, generator=g).cuda()
    b1 = R.chunkwise_backward(qc, kc, vc, d_o, gam, th, chunk=1, pos0=5, state_in=sc)
    b2 = R.chunkwise_backward(qc, kc, vc, d_o, gam, th, chunk=64, pos0=5, state_in=sc)
    assert R.sync_status() == R.RET_OK
    assert max_rel_inf(gpu_np(o1), gpu_np(o2)) < FP32_TOL and max_rel_inf(gpu_np(s1), gpu_np(s2)) < FP32_TOL
    for x, y in zip(b1, b2):
        assert max_rel_inf(gpu_np(x), gpu_np(y)) < FP32_TOL
    # rotation: 600000 rows (75000 groups of 8)
    x = torch.randn(1, 1, 600000, 8, generator=g).cuda()
    y = R.rotate(x, th, pos0=3)
    assert R.sync_status() == R.RET_OK
    tail = x[0, 0, -4:].double().cpu().numpy()
    sin, cos = O.rotation_tables(np.arange(600000 - 4, 600000) + 3, th.astype(np.float64))
    assert np.max(np.abs(gpu_np(y[0, 0, -4:]) - O.theta_shift(tail, sin, cos))) < 1e-4
    # tensor cores, chunk-parallel layout: 64 heads × 1100 chunks = 70400 rows
    w = Workload("fold", 1, 64, 1100 * 128, 64, 64, "bf16", 128, 1.0 / 8, state_std=0.1)
    inp = make_inputs(w, seed=3)
    d = _cuda(inp)
    args = (d["q"], d["k"], d["v"], inp["gamma"], inp["theta"])
    R.force_path(R.RET_PATH_TC_CARRY)   # 64 one-tile heads would otherwise pick the chunk-parallel layout
    try:
        oc, sc_ = R.chunkwise(*args, chunk=128, state_in=d["state_in"])
    finally:
        R.force_path(0)
    os_, ss = R.chunkwise(*args, chunk=128, state_in=d["state_in"], layout="scan")
    assert R.sync_status() == R.RET_OK
    assert torch.equal(oc, os_) and torch.equal(sc_, ss)


# ------------------------------------------------------------------ limits --
@pytest.mark.parametrize("case", ["widest_fp32", "most_heads_tc", "last_positions_tc", "last_positions_fp32",
                                  "no_decay_tc"])
def test_limits_vs_oracle(case):
    """The boundary's largest legal values: d_k = 512 and d_v = 1024 (fp32
    kernels), 128 heads (tensor cores), a sequence ending at position 2^24
    (the rotation at its largest angles, tensor cores), and γ = 1 (no decay:
    the state is a plain sum) next to the smallest tensor-core γ."""
    if case == "widest_fp32":
        w, inp = _custom(1, 1, 70, 512, 1024, "f32", 32, state_std=0.1, seed=5)
        pos0 = 11
    elif case == "most_heads_tc":
        w, inp = _custom(1, 128, 256, 64, 64, "bf16", 128, std=0.125, state_std=0.1, seed=6)
        pos0 = 0
    elif case == "last_positions_tc":
        w, inp = _custom(1, 2, 300, 128, 128, "bf16", 128, state_std=0.1, seed=7)
        pos0 = (1 << 24) - 300
    elif case == "last_positions_fp32":
        w, inp = _custom(1, 2, 200, 64, 32, "f32", 64, state_std=0.1, seed=9)
        pos0 = (1 << 24) - 200
    else:
        w, inp = _custom(1, 2, 384, 128, 128, "bf16", 128, std=0.5, state_std=0.1, seed=8)
        inp["gamma"] = np.array([1.0, 0.75], np.float32)   # 0.75^127 ≈ 1.4e-16 ≥ 2^-60
        pos0 = 2
    d = _cuda(inp)
    path = R.plan("chunkwise", w.torch_dtype, w.B, w.H, w.L, w.d_k, w.d_v, w.chunk, gamma=inp["gamma"])[0]
    assert path == (R.RET_PATH_SIMT if w.dtype == "f32" else R.RET_PATH_TC)
    o, s = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=w.chunk, pos0=pos0,
                       state_in=d["state_in"], out_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    ref_o, ref_s = _oracle_full(inp, w, "chunkwise", w.chunk, pos0=pos0)
    assert_close(gpu_np(o), ref_o, w.torch_dtype, f"{case} out")
    assert_close(gpu_np(s), ref_s, w.torch_dtype, f"{case} state")


def test_largest_positions_on_the_other_paths():
    """Sequences that end at position 2^24 (the largest rotation angles)
    through the decode step, the gradient pass on both paths, the parameter
    gradients and the MSR block, each against the oracle."""
    top = 1 << 24
    # decode: one token at position 2^24 − 1, fp32 inputs
    w, inp = _custom(2, 2, 1, 32, 24, "f32", 1, state_std=0.1, seed=31)
    d = _cuda(inp)
    st = d["state_in"].clone()
    o = R.step(d["q"][:, :, 0].contiguous(), d["k"][:, :, 0].contiguous(), d["v"][:, :, 0].contiguous(),
               inp["gamma"], inp["theta"], top - 1, st)
    ref_o, ref_s = O.decode_step(to_f64(inp["q"][:, :, 0]), to_f64(inp["k"][:, :, 0]), to_f64(inp["v"][:, :, 0]),
                                 inp["gamma"].astype(np.float64), inp["theta"].astype(np.float64), top - 1,
                                 to_f64(inp["state_in"]))
    assert R.sync_status() == R.RET_OK
    assert_close(gpu_np(o), ref_o, torch.float32, "decode out")
    assert_close(gpu_np(st), ref_s, torch.float32, "decode state")
    # gradient pass and parameter gradients: fp32 kernels and tensor cores
    for dtype, L, d_k, d_v, chunk in (("f32", 70, 16, 16, 16), ("bf16", 256, 128, 128, 128)):
        w, inp = _custom(1, 2, L, d_k, d_v, dtype, chunk, state_std=0.1, seed=L)
        gi = make_grad_inputs(w, seed=L + 1, d_state_std=1.0)
        d = _cuda(inp)
        p0 = top - L
        d_o, dso = gi["d_out"].cuda(), gi["d_state_out"].cuda()
        got = R.chunkwise_backward(d["q"], d["k"], d["v"], d_o, inp["gamma"], inp["theta"], chunk=chunk,
                                   pos0=p0, state_in=d["state_in"], d_state_out=dso, grad_dtype=torch.float32)
        out, _ = R.chunkwise(d["q"], d["k"], d["v"], inp["gamma"], inp["theta"], chunk=chunk, pos0=p0,
                             state_in=d["state_in"], out_dtype=torch.float32)
        dg, dt = R.param_grads(d["q"], d["k"], d["v"], d_o, out, *got[:3], inp["gamma"], inp["theta"], pos0=p0,
                               state_in=d["state_in"], d_state_out=dso)
        assert R.sync_status() == R.RET_OK
        ref = _oracle_bwd(inp, gi, p0)
        tol = torch.float32 if dtype == "f32" else torch.bfloat16
        for g, r, name in zip(got, ref, ("dq", "dk", "dv", "dS_in")):
            assert_close(gpu_np(g), r, tol, f"{dtype} {name}")
        rg, rt = O.retention_param_grads(to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"]),
                                         np.asarray(inp["gamma"], np.float64), np.asarray(inp["theta"], np.float64),
                                         p0, to_f64(inp["state_in"]), to_f64(gi["d_out"]),
                                         to_f64(gi["d_state_out"]))
        lim = 1e-4 if dtype == "f32" else BF16_TOL
        assert max_rel_inf(gpu_np(dg), rg) <= lim and max_rel_inf(gpu_np(dt), rt) <= lim, dtype
    # the MSR block (rotation in the projection epilogues)
    g = torch.Generator().manual_seed(5)
    B, L, D, H, d_k, d_v = 1, 300, 256, 2, 128, 256
    x = (torch.randn(B, L, D, generator=g)).to(torch.bfloat16)
    ws = [(torch.randn(*s, generator=g) * sc).to(torch.bfloat16) for s, sc in
          (((D, H, d_k), D ** -0.5), ((D, H, d_k), D ** -0.5), ((D, H, d_v), D ** -0.5), ((D, H, d_v), D ** -0.5),
           ((H, d_v, D), (H * d_v) ** -0.5))]
    gam, th = gamma_schedule(H), theta_schedule(d_k)
    z, _ = R.msr_block(x.cuda(), *[t.cuda() for t in ws], gam, th, pos0=top - L, out_dtype=torch.float32)
    assert R.sync_status() == R.RET_OK
    ref_z, _ = O.msr_block(to_f64(x), *[to_f64(t) for t in ws], gam.astype(np.float64), th.astype(np.float64),
                           top - L, None, 1e-5, 128)
    assert_close(gpu_np(z), ref_z, torch.bfloat16, "block z")
