"""ctypes front end of the fp64 CPU oracle (``dg_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA path never imports this module
and this module never imports the CUDA path.  Inputs are numpy arrays of the raw
bit patterns (bf16 as uint16, e4m3 as uint8); outputs are fp64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dg_oracle.c")
_LIB = os.path.join(_HERE, "libdg_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        D = ctypes.c_double
        L.dgo_e4m3_value.argtypes = [ctypes.c_uint8]
        L.dgo_e4m3_value.restype = D
        L.dgo_silu.argtypes = [D]
        L.dgo_silu.restype = D
        L.dgo_round_bf16.argtypes = [P, P, I64]
        L.dgo_bf16_to_double.argtypes = [P, P, I64]
        L.dgo_linear_bf16.argtypes = [P, P, I64, I64, P, I64, P, P]
        L.dgo_gate_up_silu.argtypes = [P, P, I64, I64, P, I64, P, P, P, P, P]
        L.dgo_head_fp8.argtypes = [P, P, D, I64, I64, P, I64, P, P]
        L.dgo_head_argmax.argtypes = [P, P, D, I64, I64, I64, P, P, P]
        L.dgo_moe_route.argtypes = [P, I64, I64, I64, P, P, P, P, P]
        L.dgo_moe_route.restype = ctypes.c_int32
        L.dgo_moe_w1_silu.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, P, P, P, P, P]
        L.dgo_moe_w2.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, P, P]
        L.dgo_e4m3_encode.argtypes = [ctypes.c_float]
        L.dgo_e4m3_encode.restype = ctypes.c_uint8
        L.dgo_a8_quant.argtypes = [P, I64, I64, P, P]
        L.dgo_a8w8_linear.argtypes = [P, P, P, P, I64, I64, P, I64, P, P]
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, n_all):
    if rows is None:
        return None, None, n_all
    r, p = _c(rows, np.int64)
    return r, p, len(r)


def e4m3_value(code: int) -> float:
    return lib().dgo_e4m3_value(int(code) & 0xFF)


def silu(g: float) -> float:
    return lib().dgo_silu(float(g))


def round_bf16(v) -> np.ndarray:
    """fp64 array -> uint16 bf16 bit patterns, round to nearest even."""
    v, pv = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().dgo_round_bf16(pv, out.ctypes.data_as(ctypes.c_void_p), v.size)
    return out


def bf16_to_double(b) -> np.ndarray:
    b, pb = _c(b, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().dgo_bf16_to_double(pb, out.ctypes.data_as(ctypes.c_void_p), b.size)
    return out


def linear_bf16(x, W, rows=None):
    """x [M,K] uint16, W [N,K] uint16 -> (y [M,nrows] f64, absdot [M,nrows] f64)."""
    x, px = _c(x, np.uint16)
    W, pW = _c(W, np.uint16)
    M, K = x.shape
    _r, pr, nr = _rows(rows, W.shape[0])
    y = np.empty((M, nr)); a = np.empty((M, nr))
    lib().dgo_linear_bf16(px, pW, M, K, pr, nr, y.ctypes.data_as(ctypes.c_void_p),
                          a.ctypes.data_as(ctypes.c_void_p))
    return y, a


def gate_up_silu(x, Wgu, cols=None):
    """-> dict(out, g, u, absg, absu), each [M, ncols] f64."""
    x, px = _c(x, np.uint16)
    Wgu, pW = _c(Wgu, np.uint16)
    M, K = x.shape
    _c_, pc, nc = _rows(cols, Wgu.shape[0] // 2)
    res = {k: np.empty((M, nc)) for k in ("out", "g", "u", "absg", "absu")}
    lib().dgo_gate_up_silu(px, pW, M, K, pc, nc, *[res[k].ctypes.data_as(ctypes.c_void_p)
                                                   for k in ("out", "g", "u", "absg", "absu")])
    return res


def head_fp8(x, Wq, scale: float, rows=None):
    """-> (logit [M,nrows] f64, absdot [M,nrows] f64)."""
    x, px = _c(x, np.uint16)
    Wq, pW = _c(Wq, np.uint8)
    M, K = x.shape
    _r, pr, nr = _rows(rows, Wq.shape[0])
    lg = np.empty((M, nr)); a = np.empty((M, nr))
    lib().dgo_head_fp8(px, pW, float(scale), M, K, pr, nr, lg.ctypes.data_as(ctypes.c_void_p),
                       a.ctypes.data_as(ctypes.c_void_p))
    return lg, a


def head_argmax(x, Wq, scale: float):
    """-> (idx [M] int32, best [M] f32, gap [M] f64)."""
    x, px = _c(x, np.uint16)
    Wq, pW = _c(Wq, np.uint8)
    M, K = x.shape
    N = Wq.shape[0]
    idx = np.empty(M, np.int32); best = np.empty(M, np.float32); gap = np.empty(M)
    lib().dgo_head_argmax(px, pW, float(scale), M, N, K, idx.ctypes.data_as(ctypes.c_void_p),
                          best.ctypes.data_as(ctypes.c_void_p), gap.ctypes.data_as(ctypes.c_void_p))
    return idx, best, gap


def moe_route(ids, E: int):
    """-> dict(valid [M,topk], experts [U], offsets [U+1], pair_tok [P], pair_slot [P])."""
    ids, pi = _c(ids, np.int32)
    M, topk = ids.shape
    valid = np.empty((M, topk), np.int32)
    experts = np.empty(E, np.int32); offsets = np.empty(E + 1, np.int32)
    ptok = np.empty(M * topk, np.int32); pslot = np.empty(M * topk, np.int32)
    U = lib().dgo_moe_route(pi, M, topk, E, *[a.ctypes.data_as(ctypes.c_void_p)
                                              for a in (valid, experts, offsets, ptok, pslot)])
    P = int(offsets[U])
    return dict(valid=valid, experts=experts[:U].copy(), offsets=offsets[:U + 1].copy(),
                pair_tok=ptok[:P].copy(), pair_slot=pslot[:P].copy())


def moe_w1_silu(x, ids, W1q, s1):
    """x [M,K] u16, ids [M,topk] i32, W1q [E,2I,K] u8, s1 [E,2I] f32 -> dict of [M,topk,I] f64."""
    x, px = _c(x, np.uint16)
    ids, pi = _c(ids, np.int32)
    W1q, pW = _c(W1q, np.uint8)
    s1, ps = _c(s1, np.float32)
    M, K = x.shape
    topk = ids.shape[1]
    E, twoI, _ = W1q.shape
    I = twoI // 2
    res = {k: np.empty((M, topk, I)) for k in ("a", "g", "u", "absg", "absu")}
    lib().dgo_moe_w1_silu(px, pi, pW, ps, M, topk, E, I, K,
                          *[res[k].ctypes.data_as(ctypes.c_void_p) for k in ("a", "g", "u", "absg", "absu")])
    return res


def moe_w2(a, ids, gw, W2q, s2):
    """a [M,topk,I] u16, ids [M,topk], gw [M,topk] f32, W2q [E,Nout,I] u8, s2 [E,Nout]
    -> (y [M,Nout] f64, absdot [M,Nout] f64)."""
    a, pa = _c(a, np.uint16)
    ids, pi = _c(ids, np.int32)
    gw, pg = _c(gw, np.float32)
    W2q, pW = _c(W2q, np.uint8)
    s2, ps = _c(s2, np.float32)
    M, topk = ids.shape
    E, Nout, I = W2q.shape
    y = np.empty((M, Nout)); b = np.empty((M, Nout))
    lib().dgo_moe_w2(pa, pi, pg, pW, ps, M, topk, E, I, Nout, y.ctypes.data_as(ctypes.c_void_p),
                     b.ctypes.data_as(ctypes.c_void_p))
    return y, b


def e4m3_encode(v: float) -> int:
    """Nearest e4m3 code (ties to even, saturating at 448) of a binary32 value."""
    return int(lib().dgo_e4m3_encode(float(v)))


def a8_quant(x):
    """x [M,K] uint16 bf16 bits -> (q [M,K] uint8 e4m3 codes, sx [M, ceil(K/128)] float32)."""
    x, px = _c(x, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    sx = np.empty((M, (K + 127) // 128), np.float32)
    lib().dgo_a8_quant(px, M, K, q.ctypes.data_as(ctypes.c_void_p), sx.ctypes.data_as(ctypes.c_void_p))
    return q, sx


def a8w8_linear_q(q, sx, Wq, sw, rows=None):
    """Block-scaled product of quantised activations: -> (y [M,nrows] f64, absdot [M,nrows] f64)."""
    q, pq = _c(q, np.uint8)
    sx, psx = _c(sx, np.float32)
    Wq, pW = _c(Wq, np.uint8)
    sw, psw = _c(sw, np.float32)
    M, K = q.shape
    _r, pr, nr = _rows(rows, Wq.shape[0])
    y = np.empty((M, nr)); a = np.empty((M, nr))
    lib().dgo_a8w8_linear(pq, psx, pW, psw, M, K, pr, nr, y.ctypes.data_as(ctypes.c_void_p),
                          a.ctypes.data_as(ctypes.c_void_p))
    return y, a


def a8w8_linear(x, Wq, sw, rows=None):
    """The whole A8W8 step on bf16 activations: quantise, then the block-scaled product.
    -> dict(y, absdot, q, sx)."""
    q, sx = a8_quant(x)
    y, a = a8w8_linear_q(q, sx, Wq, sw, rows)
    return {"y": y, "absdot": a, "q": q, "sx": sx}
