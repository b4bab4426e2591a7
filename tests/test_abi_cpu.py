"""Host-side checks of the C ABI: build, symbol exports, validation, planning.

None of these launch a kernel, so they run without a GPU.
"""

import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

from linear_recurrent_sequence_prologue_b300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "retention.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ret_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("ret_parallel", "ret_chunkwise", "ret_step", "ret_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (ret_[a-z_0-9]+)\b", out))
    missing = [n for n in header_functions() if n not in exported]
    assert not missing, missing
    for n in header_functions():
        assert hasattr(lib, n)
        assert n in _lib.SIGNATURES, f"binding lacks a signature for {n}"


def test_status_strings_and_version(lib):
    assert lib.ret_abi_version() == 1
    for code in range(6):
        assert lib.ret_status_string(code)
    assert b"unknown" in lib.ret_status_string(99)


def _fp(a):
    return a.ctypes.data_as(C.POINTER(C.c_float))


def _chunkwise_args(**over):
    g = np.full(2, 0.9, np.float32)
    t = np.ones(8, np.float32)
    a = dict(q=C.c_void_p(0x1000), k=C.c_void_p(0x2000), v=C.c_void_p(0x3000), in_dt=_lib.RET_F32,
             gamma=_fp(g), theta=_fp(t), B=1, H=2, L=64, d_k=16, d_v=16, pos0=0, chunk=16,
             s_in=None, s_out=None, out=C.c_void_p(0x4000), out_dt=_lib.RET_F32, gn=None,
             ws=None, wsb=0, stream=None)
    a.update(over)
    return a, (g, t)


def _call_chunkwise(lib, a):
    return lib.ret_chunkwise(a["q"], a["k"], a["v"], a["in_dt"], a["gamma"], a["theta"], a["B"],
                             a["H"], a["L"], a["d_k"], a["d_v"], a["pos0"], a["chunk"], a["s_in"],
                             a["s_out"], a["out"], a["out_dt"], a["gn"], a["ws"], a["wsb"],
                             a["stream"])


@pytest.mark.parametrize("over,expect", [
    (dict(q=None), _lib.RET_EINVAL),
    (dict(out=None), _lib.RET_EINVAL),
    (dict(q=C.c_void_p(0x1004)), _lib.RET_EINVAL),          # misaligned
    (dict(d_k=15), _lib.RET_EINVAL),                          # odd d_k
    (dict(d_k=1024), _lib.RET_EINVAL),
    (dict(H=0), _lib.RET_EINVAL),
    (dict(H=129), _lib.RET_EINVAL),
    (dict(L=0), _lib.RET_EINVAL),
    (dict(chunk=0), _lib.RET_EINVAL),
    (dict(pos0=-1), _lib.RET_EINVAL),
    (dict(pos0=(1 << 24) - 10), _lib.RET_EINVAL),            # positions beyond 2^24
    (dict(in_dt=7), _lib.RET_EINVAL),
    (dict(gamma=None), _lib.RET_EINVAL),
    (dict(ws=None, wsb=0), _lib.RET_EWORKSPACE),              # fp32 path needs scratch
])
def test_chunkwise_validation_is_synchronous(lib, over, expect):
    a, keep = _chunkwise_args(**over)
    assert _call_chunkwise(lib, a) == expect


def test_gamma_out_of_range_rejected(lib):
    for bad in (0.0, -0.5, 1.5, float("nan")):
        g = np.array([0.9, bad], np.float32)
        a, keep = _chunkwise_args(gamma=_fp(g))
        assert _call_chunkwise(lib, a) == _lib.RET_EINVAL


def test_step_and_rotate_validation(lib):
    g = np.full(2, 0.9, np.float32)
    t = np.ones(8, np.float32)
    st = lib.ret_step(None, None, None, _lib.RET_BF16, _fp(g), _fp(t), 1, 2, 16, 16, 0,
                      C.c_void_p(0x1000), C.c_void_p(0x2000), _lib.RET_BF16, None, None)
    assert st == _lib.RET_EINVAL
    st = lib.ret_rotate(C.c_void_p(0x1000), _lib.RET_BF16, _fp(t), 1, 1, 8, 15, 0, 1.0,
                        C.c_void_p(0x2000), _lib.RET_BF16, None)
    assert st == _lib.RET_EINVAL
    assert lib.ret_selftest_timeout(0, None) == _lib.RET_EINVAL
    assert lib.ret_force_path(5) == _lib.RET_EINVAL
    # the one-CTA tensor-core variant is selectable; plans still report the tensor-core path
    assert lib.ret_force_path(_lib.RET_PATH_TC_SINGLE) == _lib.RET_OK
    try:
        assert _plan(lib, _lib.RET_BF16, 2, 16, 8192, 256, 512, 128)[0] == _lib.RET_PATH_TC
    finally:
        assert lib.ret_force_path(0) == _lib.RET_OK


def test_rowpos_validation(lib):
    """ret_chunkwise_rowpos checks its per-row start positions before any launch."""
    g = np.full(2, 0.99, np.float32)
    t = np.ones(8, np.float32)
    fp = lambda a: a.ctypes.data_as(C.POINTER(C.c_float))
    P = C.c_void_p(0x1000)

    def call(rows, B=2):
        arr = None if rows is None else (C.c_int64 * len(rows))(*rows)
        return lib.ret_chunkwise_rowpos(P, P, P, _lib.RET_F32, fp(g), fp(t), B, 2, 64, 16, 16, arr, 16,
                                        None, None, P, _lib.RET_F32, None, None, 0, None)

    assert call(None) == _lib.RET_EINVAL                      # no array
    assert call([0, -1]) == _lib.RET_EINVAL                   # negative start
    assert call([0, (1 << 24) - 10]) == _lib.RET_EINVAL       # positions past 2^24
    assert call([0] * 300, B=300) == _lib.RET_EUNSUPPORTED    # more rows than the constant block holds
    assert call([0, 5]) == _lib.RET_EWORKSPACE                # valid: stops at the missing workspace


def _plan(lib, in_dt, B, H, L, d_k, d_v, chunk, gn=0, gamma=None):
    path, nb = C.c_int(0), C.c_size_t(0)
    gp = _fp(gamma) if gamma is not None else None
    st = lib.ret_chunkwise_plan(in_dt, gp, B, H, L, d_k, d_v, chunk, in_dt, gn, C.byref(path), C.byref(nb))
    assert st == _lib.RET_OK
    return path.value, nb.value


def _ring_bytes(heads, L, d_k):
    """Workspace of the carried layout on CTA pairs: the ring's counters (256 B),
    4 chunk slots of Q″ and of K̂′ per head of one launch (bf16), the
    (cos, sin) table [L][d_k/2]."""
    return 256 + 2 * heads * 4 * 128 * d_k * 2 + L * (d_k // 2) * 8


def _plan_compact(lib, in_dt, B, H, L, d_k, d_v, chunk, gn=0):
    path, nb = C.c_int(0), C.c_size_t(0)
    st = lib.ret_chunkwise_plan_compact(in_dt, None, B, H, L, d_k, d_v, chunk, in_dt, gn, C.byref(path),
                                        C.byref(nb))
    assert st == _lib.RET_OK
    return path.value, nb.value


def test_path_selection(lib):
    # 7B shape: tensor-core path, workspace = rotated Q′ and K̂′ in bf16
    front = 2 * 2 * 16 * 8192 * 256 * 2
    assert _plan(lib, _lib.RET_BF16, 2, 16, 8192, 256, 512, 128) == (_lib.RET_PATH_TC, front)
    # the compact mode: 32 heads (128 consumer CTAs) per launch in the ring
    assert _plan_compact(lib, _lib.RET_BF16, 2, 16, 8192, 256, 512, 128) == \
        (_lib.RET_PATH_TC, _ring_bytes(32, 8192, 256))
    nb = front
    # the chunk-parallel layout (front pass) adds one fp32 d_k×d_v state per (b, h, chunk)
    path, nb2 = C.c_int(0), C.c_size_t(0)
    assert lib.ret_chunkwise_scan_plan(_lib.RET_BF16, None, 2, 16, 8192, 256, 512, 128,
                                       _lib.RET_BF16, 0, C.byref(path), C.byref(nb2)) == _lib.RET_OK
    assert path.value == _lib.RET_PATH_TC
    assert nb2.value == front + 2 * 16 * 64 * 256 * 512 * 4
    # the parallel form of the same shape runs on the tensor cores as well
    assert lib.ret_parallel_plan(_lib.RET_BF16, None, 2, 16, 8192, 256, 512, _lib.RET_BF16, 0, 0,
                                 C.byref(path), C.byref(nb2)) == _lib.RET_OK
    assert path.value == _lib.RET_PATH_TC and nb2.value == front   # rotated Q′ / K̂′ only
    # the ring holds at most 128 consumer CTAs' heads: 64 at d_v = 256, fewer when B·H is smaller
    assert _plan_compact(lib, _lib.RET_BF16, 8, 16, 2048, 256, 256, 128)[1] == _ring_bytes(64, 2048, 256)
    assert _plan_compact(lib, _lib.RET_BF16, 1, 3, 1300, 128, 256, 128)[1] == \
        _ring_bytes(3, 1300, 128) + 3 * 128 * 256 * 4
    # sequences of no more chunks than the ring holds: the front pass is smaller
    assert _plan_compact(lib, _lib.RET_BF16, 2, 16, 512, 256, 512, 128) == \
        _plan(lib, _lib.RET_BF16, 2, 16, 512, 256, 512, 128) == (_lib.RET_PATH_TC, 2 * 2 * 16 * 512 * 256 * 2)
    # few CTAs walking many chunks (4 carried CTAs, 32 chunks: 6·1 + 8 < 32): the
    # chunk-parallel layout, whose workspace adds the per-chunk states
    assert _plan(lib, _lib.RET_BF16, 1, 2, 4096, 256, 512, 128) == \
        (_lib.RET_PATH_TC, 2 * 2 * 4096 * 256 * 2 + 2 * 32 * 256 * 512 * 4)
    assert lib.ret_force_path(_lib.RET_PATH_TC_CARRY) == _lib.RET_OK
    try:   # the carried layout kept: the rotated Q′ / K̂′ only
        assert _plan(lib, _lib.RET_BF16, 1, 2, 4096, 256, 512, 128) == (_lib.RET_PATH_TC, 2 * 2 * 4096 * 256 * 2)
    finally:
        assert lib.ret_force_path(0) == _lib.RET_OK
    # …but not for few chunks (4 CTAs, 4 chunks) or many one-chunk CTAs: the Small
    # MSR workload (d_v = 64, one 128-wide tile of which 64 columns are live;
    # chunk 64 runs on the 128-token tile: 32 CTAs × 16 chunks, 6·4 + 8 ≥ 16)
    assert _plan(lib, _lib.RET_BF16, 2, 2, 512, 256, 512, 128) == (_lib.RET_PATH_TC, 2 * 2 * 2 * 512 * 256 * 2)
    assert _plan(lib, _lib.RET_BF16, 4, 8, 2048, 64, 64, 64) == (_lib.RET_PATH_TC, 2 * 32 * 2048 * 64 * 2)
    # no compact mode off the CTA-pair shapes: the same bytes as the plan
    assert _plan_compact(lib, _lib.RET_BF16, 2, 2, 512, 64, 128, 128) == \
        _plan(lib, _lib.RET_BF16, 2, 2, 512, 64, 128, 128)
    assert _plan_compact(lib, _lib.RET_F32, 1, 2, 64, 16, 16, 16) == _plan(lib, _lib.RET_F32, 1, 2, 64, 16, 16, 16)
    # a length that is not a multiple of the chunk stays on the tensor cores, with
    # the rotated Q′ / K̂′ padded to whole chunks; the parallel form needs whole blocks
    p, nb = _plan(lib, _lib.RET_BF16, 2, 16, 8000, 256, 512, 128)
    # (+ an fp32 staging tile of 128 rows per sequence for the short last chunk's outputs)
    assert p == _lib.RET_PATH_TC and nb == 2 * 2 * 16 * 8064 * 256 * 2 + 2 * 16 * 128 * 512 * 4
    assert _plan_compact(lib, _lib.RET_BF16, 2, 16, 8000, 256, 512, 128)[1] == \
        _ring_bytes(32, 8000, 256) + 2 * 16 * 128 * 512 * 4
    assert lib.ret_parallel_plan(_lib.RET_BF16, None, 2, 16, 8000, 256, 512, _lib.RET_BF16, 0, 0,
                                 C.byref(path), C.byref(nb2)) == _lib.RET_OK
    assert path.value == _lib.RET_PATH_SIMT
    assert _plan(lib, _lib.RET_F32, 1, 2, 64, 16, 16, 16)[0] == _lib.RET_PATH_SIMT
    assert _plan(lib, _lib.RET_BF16, 4, 8, 2048, 64, 64, 32)[0] == _lib.RET_PATH_SIMT   # chunk 32
    assert _plan(lib, _lib.RET_BF16, 4, 8, 2048, 64, 96, 64)[0] == _lib.RET_PATH_SIMT   # d_v 96
    # a head whose γ^127 underflows the rewritten form goes to the fp32 kernels
    g = np.array([0.5, 0.99], np.float32)
    assert _plan(lib, _lib.RET_BF16, 1, 2, 256, 256, 128, 128, gamma=g)[0] == _lib.RET_PATH_SIMT
    g = np.array([0.9, 0.99], np.float32)
    assert _plan(lib, _lib.RET_BF16, 1, 2, 256, 256, 128, 128, gamma=g)[0] == _lib.RET_PATH_TC


def test_backward_plan_and_validation(lib):
    """ret_chunkwise_backward: workspace layout and synchronous argument checks."""
    path, nb = C.c_int(0), C.c_size_t(0)

    def plan(in_dt, B, H, L, d_k, d_v, chunk, gamma=None):
        st = lib.ret_chunkwise_backward_plan(in_dt, _fp(gamma) if gamma is not None else None, B, H, L,
                                             d_k, d_v, chunk, C.byref(path), C.byref(nb))
        assert st == _lib.RET_OK
        return path.value, nb.value

    BH, L = 32, 8192
    rk, rv = BH * L * 256 * 4, BH * L * 512 * 4
    # tensor cores, the operands of the three evaluations in bf16: ω·dO and ζ·V
    # (d_v wide, shared by the dQ′ and dK′ evaluations), K̂′ and Q″ (d_k wide),
    # all padded to whole chunks; K′ and Q′ (the values of dQ′ and dK′, once);
    # then fp32 outputs (two pieces of d_k), one prepared state, the (cos, sin)
    # table of the rotation and, for a ragged length, a staging tile
    def tc_bytes(Lx, Lpx, tail):
        up = lambda n: -(-n // 256) * 256
        return (2 * BH * Lpx * 512 * 2 + 2 * BH * Lpx * 256 * 2 + 2 * BH * Lx * 256 * 2
                + BH * Lx * 512 * 4 + BH * 256 * 512 * 4 + up(Lx * 128 * 8)
                + (BH * 128 * 512 * 4 if tail else 0))

    assert plan(_lib.RET_BF16, 2, 16, 8192, 256, 512, 128) == (_lib.RET_PATH_TC, tc_bytes(8192, 8192, False))
    # a ragged length pads the folded operands to whole chunks and adds a staging tile
    assert plan(_lib.RET_BF16, 2, 16, 8000, 256, 512, 128) == (_lib.RET_PATH_TC, tc_bytes(8000, 8064, True))
    # fp32 kernels: Q′↓, K′, K′↓ (fp32); dO, V in order (bf16 inputs only) and
    # reversed; one evaluation output; per-chunk states; one prepared state
    simt = 3 * rk + 4 * rv + rv + BH * 64 * 256 * 512 * 4 + BH * 256 * 512 * 4
    assert plan(_lib.RET_BF16, 2, 16, 8192, 256, 512, 64)[0] == _lib.RET_PATH_SIMT      # chunk 64
    assert plan(_lib.RET_BF16, 2, 16, 8192, 64, 512, 128)[0] == _lib.RET_PATH_SIMT      # d_k 64
    g = np.array([0.74] + [0.99] * 15, np.float32)   # the reverse evaluations' γ^-255 > 2^100
    assert plan(_lib.RET_BF16, 2, 16, 8192, 256, 512, 128, gamma=g)[0] == _lib.RET_PATH_SIMT
    g = np.array([0.5] + [0.99] * 15, np.float32)                                         # γ^127 underflows
    assert plan(_lib.RET_BF16, 2, 16, 8192, 256, 512, 128, gamma=g) == (_lib.RET_PATH_SIMT, simt)
    assert lib.ret_force_path(_lib.RET_PATH_SIMT) == _lib.RET_OK
    try:
        assert plan(_lib.RET_BF16, 2, 16, 8192, 256, 512, 128) == (_lib.RET_PATH_SIMT, simt)
    finally:
        assert lib.ret_force_path(0) == _lib.RET_OK
    assert plan(_lib.RET_F32, 2, 16, 8192, 256, 512, 128) == (_lib.RET_PATH_SIMT, simt - 2 * rv)
    assert lib.ret_chunkwise_backward_plan(_lib.RET_F32, None, 1, 1, 8, 16, 16, 0,
                                           C.byref(path), C.byref(nb)) == _lib.RET_EINVAL

    g = np.full(2, 0.9, np.float32)
    t = np.ones(8, np.float32)
    P, M = C.c_void_p(0x1000), C.c_void_p(0x1008)

    def call(d_out=P, dk=P, gamma=g, B=1, H=2, L=64, chunk=16, ws=None, wsn=0):
        return lib.ret_chunkwise_backward(P, P, P, d_out, _lib.RET_F32, _fp(gamma), _fp(t), B, H, L, 16,
                                          16, 0, chunk, None, None, P, dk, P, _lib.RET_F32, None, ws,
                                          wsn, None)

    assert call(d_out=None) == _lib.RET_EINVAL                       # no upstream gradient
    assert call(dk=M) == _lib.RET_EINVAL                             # misaligned output
    assert call(chunk=0) == _lib.RET_EINVAL
    assert call(gamma=np.array([0.9, 1.5], np.float32)) == _lib.RET_EINVAL
    assert call(gamma=np.array([0.9, 2.0 ** -70], np.float32)) == _lib.RET_EUNSUPPORTED
    gh = np.full(128, 0.9, np.float32)
    # 128 heads × 1024 chunks of 64: more (b, h, chunk) rows than one grid
    # dimension holds, folded over two, so only the workspace is missing
    assert call(gamma=gh, H=128, L=65536, chunk=64) == _lib.RET_EWORKSPACE
    assert call(gamma=gh, B=512, H=128, L=1) == _lib.RET_EUNSUPPORTED        # B·H > 65535
    assert call() == _lib.RET_EWORKSPACE                             # valid: no workspace
    assert call(ws=P, wsn=16) == _lib.RET_EWORKSPACE                 # too small


def test_decay_row_norm_validation(lib):
    """ret_decay_row_norm checks its arguments before any launch."""
    g = np.array([0.9, 0.99], np.float32)
    P = C.c_void_p(0x1000)

    def call(out=P, gamma=g, H=2, L=8, pos0=0, dt=_lib.RET_F32):
        return lib.ret_decay_row_norm(out, dt, _fp(gamma), 1, H, L, 16, pos0, None)

    assert call(out=None) == _lib.RET_EINVAL
    assert call(out=C.c_void_p(0x1004)) == _lib.RET_EINVAL                 # misaligned
    assert call(gamma=np.array([0.9, 1.01], np.float32)) == _lib.RET_EINVAL
    assert call(gamma=np.array([0.9, 0.0], np.float32)) == _lib.RET_EINVAL
    assert call(pos0=-1) == _lib.RET_EINVAL
    assert call(pos0=(1 << 24) - 4) == _lib.RET_EINVAL                     # positions past 2^24
    assert call(dt=7) == _lib.RET_EINVAL


def test_chunk_size_policy(lib):
    """128 where the tensor-core path applies, else round(√L) (at least 1)."""
    def b(dt, L, d_k=256, d_v=512, H=16, gamma=None):
        return lib.ret_chunk_size(dt, _fp(gamma) if gamma is not None else None, H, L, d_k, d_v)

    assert b(_lib.RET_BF16, 8192) == 128                  # 7B shape: the tensor-core tile
    assert b(_lib.RET_BF16, 8000) == 128                  # ragged lengths stay on the tile
    assert b(_lib.RET_F32, 8192) == 91                    # √8192 = 90.5
    assert b(_lib.RET_F32, 2048, 64, 64, 8) == 45         # √2048 = 45.3
    assert b(_lib.RET_BF16, 4096, 512, 512) == 64         # d_k outside the tensor-core shapes
    assert b(_lib.RET_BF16, 4096, 256, 96) == 64          # d_v not a multiple of 128
    assert b(_lib.RET_F32, 1, 16, 16, 1) == 1
    assert b(_lib.RET_F32, 2, 16, 16, 1) == 1
    g = np.array([0.5] + [0.99] * 15, np.float32)         # γ^127 underflows the rewritten form
    assert b(_lib.RET_BF16, 8192, gamma=g) == 91
    assert b(_lib.RET_F32, 0) == 0 and b(7, 64) == 0      # invalid arguments
    assert b(_lib.RET_F32, 64, gamma=np.array([1.5] * 16, np.float32)) == 0


def test_msr_block_and_matmul_validation(lib):
    """ret_msr_block / ret_matmul: workspace layout and synchronous checks."""
    nb = C.c_size_t(0)
    g = np.full(16, 0.99, np.float32)
    assert lib.ret_msr_block_plan(_fp(g), 2, 8192, 4096, 16, 256, 512, 4096, C.byref(nb)) == _lib.RET_OK
    M, HV = 2 * 8192, 16 * 512
    core = 2 * 2 * 16 * 8192 * 256 * 2                  # Q″ and K̂′ from the projection epilogues
    assert nb.value == core + 8192 * 128 * 8 + M * HV * (2 + 4 + 2 + 2)   # table, v, fp32 o, gate, gated rows
    # shapes outside the tensor-core core or the GEMM tiling
    for args in ((2, 8192, 4000, 16, 256, 512, 4096),      # D not a multiple of 64
                 (2, 8192, 4096, 16, 256, 512, 4000),      # D_out not a multiple of 256
                 (2, 8192, 4096, 16, 512, 512, 4096),      # d_k outside the tensor-core shapes
                 (2, 8192, 4096, 3, 64, 64, 4096)):        # H·d_k not a multiple of 256
        h = args[3]
        assert lib.ret_msr_block_plan(_fp(np.full(h, 0.99, np.float32)), *args, C.byref(nb)) == \
            _lib.RET_EUNSUPPORTED
    assert lib.ret_msr_block_plan(_fp(g), 2, 8192, 4096, 16, 256, 512, 4096, None) == _lib.RET_EINVAL
    P = C.c_void_p(0x1000)
    t = np.ones(128, np.float32)
    call = lambda **kw: lib.ret_msr_block(*[kw.get(n, P) for n in ("x", "wq", "wk", "wv", "wg", "wo")],
                                          _fp(g), _fp(t), 2, 8192, 4096, 16, 256, 512, 4096, 0, None, None,
                                          kw.get("z", P), _lib.RET_BF16, kw.get("eps", 1e-5), None, 0, None)
    assert call(x=None) == _lib.RET_EINVAL
    assert call(wo=C.c_void_p(0x1008)) == _lib.RET_EINVAL          # misaligned
    assert call(eps=0.0) == _lib.RET_EINVAL
    assert call() == _lib.RET_EWORKSPACE                           # valid: no workspace
    # the GEMM alone
    assert lib.ret_matmul(None, P, P, _lib.RET_F32, 300, 512, 192, None) == _lib.RET_EINVAL
    assert lib.ret_matmul(P, P, P, _lib.RET_F32, 300, 500, 192, None) == _lib.RET_EUNSUPPORTED
    assert lib.ret_matmul(P, P, P, _lib.RET_F32, 300, 512, 100, None) == _lib.RET_EUNSUPPORTED
    assert lib.ret_matmul(P, P, P, 7, 300, 512, 192, None) == _lib.RET_EINVAL


def test_param_grads_and_groupnorm_validation(lib):
    """ret_chunkwise_param_grads, ret_groupnorm and ret_groupnorm_backward
    check their arguments (and workspace) before any launch; the plans give
    the documented sizes."""
    P, P2, P3 = C.c_void_p(0x1000), C.c_void_p(0x2000), C.c_void_p(0x3000)
    g = np.array([0.9, 0.99], np.float32)
    nb = C.c_size_t(0)
    assert lib.ret_chunkwise_param_grads_plan(2, 2, 100, 64, 32, C.byref(nb)) == _lib.RET_OK
    # 8 row segments (2 per head) and 4 walk tiles: doubles, 32 pair sums per
    # segment, the angle table (100 × 32 float2), one chunk of 64 × 64 fp32
    # states per tile, the walk partials
    assert nb.value == 256 + 1024 + 25600 + 4 * 16384 + 256 + 512
    # d_k = d_v = 128: the same parts for 16 walk tiles, plus the walks' operands
    # qb and kf as fp32, or as bf16 hi + lo rows padded to whole chunks of 128
    assert lib.ret_chunkwise_param_grads_plan(2, 2, 100, 128, 128, C.byref(nb)) == _lib.RET_OK
    assert nb.value == 256 + 2048 + 51200 + 16 * 16384 + 256 + 2048 + 2 * (4 * 128 * 128 * 4)
    assert lib.ret_chunkwise_param_grads_plan(2, 2, 100, 63, 32, C.byref(nb)) == _lib.RET_EINVAL
    th = np.full(32, 0.1, np.float32)

    def call(d_gamma=P, d_theta=P, gamma=g, d_k=64, pos0=0, ws=P, wsn=1 << 20, dq=P, in_dt=_lib.RET_BF16,
             theta=th, out=P):
        return lib.ret_chunkwise_param_grads(P, P, P, P, in_dt, out, _lib.RET_BF16, dq, P, P, _lib.RET_F32,
                                             _fp(gamma), _fp(theta), 2, 2, 100, d_k, 32, pos0, None, None,
                                             d_gamma, d_theta, ws, wsn, None)

    assert call(d_gamma=None, d_theta=None) == _lib.RET_EINVAL
    assert call(d_k=63) == _lib.RET_EINVAL
    assert call(gamma=np.array([0.9, 0.0], np.float32)) == _lib.RET_EINVAL
    assert call(theta=np.full(32, np.nan, np.float32)) == _lib.RET_EINVAL
    assert call(pos0=(1 << 24) - 50) == _lib.RET_EINVAL
    assert call(dq=None) == _lib.RET_EINVAL                      # dθ needs dq
    assert call(dq=None, d_theta=None, ws=None) == _lib.RET_EWORKSPACE   # …dγ alone does not
    assert call(out=None, d_gamma=None, ws=None) == _lib.RET_EWORKSPACE  # …and dθ needs no out
    assert call(dq=C.c_void_p(0x1008)) == _lib.RET_EINVAL       # misaligned
    assert call(in_dt=5) == _lib.RET_EINVAL
    assert call(ws=None) == _lib.RET_EWORKSPACE
    assert call(wsn=100) == _lib.RET_EWORKSPACE

    gn = _lib.RetGN(1, 1e-5, None, None)
    assert lib.ret_groupnorm(P, _lib.RET_F32, P2, _lib.RET_BF16, 1, 2, 8, 0, C.byref(gn), None) == _lib.RET_EINVAL
    gmis = _lib.RetGN(1, 1e-5, C.c_void_p(0x1004), None)       # weights read as 16-byte vectors
    assert lib.ret_groupnorm(P, _lib.RET_F32, P2, _lib.RET_BF16, 1, 2, 8, 16, C.byref(gmis), None) == \
        _lib.RET_EINVAL
    assert lib.ret_groupnorm(P, _lib.RET_F32, P, _lib.RET_BF16, 1, 2, 8, 16, C.byref(gn), None) == \
        _lib.RET_EINVAL                                          # in place needs one type
    assert lib.ret_groupnorm(P, _lib.RET_F32, P2, _lib.RET_F32, 1, 2, 8, 16, None, None) == _lib.RET_EINVAL
    bad = _lib.RetGN(1, 0.0, None, None)
    assert lib.ret_groupnorm(P, _lib.RET_F32, P2, _lib.RET_F32, 1, 2, 8, 16, C.byref(bad), None) == \
        _lib.RET_EINVAL

    assert lib.ret_groupnorm_backward_plan(2, 2, 100, 48, C.byref(nb)) == _lib.RET_OK
    assert nb.value == 2 * 2 * 2 * 2 * 48 * 4                  # [blocks][2][d_v] floats

    def gcall(x=P, dx=P3, eps=1e-5, d_v=48, dw=None, ws=None, wsn=0):
        return lib.ret_groupnorm_backward(x, P2, _lib.RET_F32, None, eps, 2, 2, 100, d_v, dx, _lib.RET_F32,
                                          dw, None, ws, wsn, None)

    assert gcall(dx=P) == _lib.RET_EINVAL                       # d_x aliases x
    assert gcall(eps=0.0) == _lib.RET_EINVAL
    assert gcall(d_v=1025) == _lib.RET_EINVAL
    assert gcall(x=C.c_void_p(0x1004)) == _lib.RET_EINVAL
    assert gcall(dw=P) == _lib.RET_EWORKSPACE                   # parameter sums need the workspace
    assert gcall(dw=P, ws=P, wsn=100) == _lib.RET_EWORKSPACE
