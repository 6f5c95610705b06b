"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one oracle function to a fixed point outside it: exact rational
brute force on tiny shapes, closed forms, identities and special cases, a
library routine, or the published OCP E4M3 table points in tests/golden.
Shapes are deliberately non-square so that a transposed operand, a swapped
gate/up row, a dropped term or a wrong sign fails at least one of them.
"""
import math
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
import torch

from oracle import oracle as O
from synth import decode_inputs as S
from tests._exact import (bf16_bits, bf16_bits_of_exact, bf16_float, e4m3_float_lib, frac,
                          rne_bf16_exact)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
mpmath.mp.dps = 50


def _silu_mp(g: Fraction) -> float:
    gm = mpmath.mpf(g.numerator) / g.denominator
    return float(gm / (1 + mpmath.exp(-gm)))


# ---------------------------------------------------------------- e4m3 decode

def test_e4m3_ocp_table_points():
    with open(os.path.join(GOLDEN, "e4m3_ocp_points.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for code, val in rows:
        got = O.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(Fraction(val)), (code, got, val)
            if val.startswith("-"):
                assert math.copysign(1.0, got) < 0


def test_e4m3_all_256_codes_match_library_decode():
    lib = e4m3_float_lib(np.arange(256))
    for c in range(256):
        got = O.e4m3_value(c)
        if math.isnan(lib[c]):
            assert math.isnan(got), c
        else:
            assert got == lib[c] and math.copysign(1, got) == math.copysign(1, lib[c]), c


def test_e4m3_positive_codes_strictly_increase_and_negate():
    vals = [O.e4m3_value(c) for c in range(0x7F)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    for c in range(1, 0x7F):
        assert O.e4m3_value(c | 0x80) == -O.e4m3_value(c)


# ---------------------------------------------------------------- bf16 rounding

def test_round_bf16_matches_torch_on_binary32_values():
    g = torch.Generator().manual_seed(7)
    v = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp2(
        torch.randint(-140, 120, (20000,), generator=g).float())
    ref = bf16_bits(v.to(torch.bfloat16))
    got = O.round_bf16(v.double().numpy())
    assert np.array_equal(got, ref)


def test_round_bf16_ties_and_double_rounding():
    one = 1.0
    cases = {
        one + 2.0 ** -8: 0x3F80,               # halfway, even neighbour is 1.0
        one + 3 * 2.0 ** -8: 0x3F82,           # halfway, rounds up to the even 1+2^-6
        one + 2.0 ** -8 + 2.0 ** -40: 0x3F81,  # just above halfway (a binary32 detour gives 1.0)
        -(one + 2.0 ** -8 + 2.0 ** -40): 0xBF81,
        2.0 ** -133: 0x0001,                   # smallest bf16 subnormal
        2.0 ** -134: 0x0000,                   # half of it: tie to even zero
    }
    got = O.round_bf16(np.array(list(cases.keys())))
    assert [int(v) for v in got] == list(cases.values())


# ---------------------------------------------------------------- linear

@pytest.mark.parametrize("M,N,K,seed", [(1, 7, 24, 1), (3, 5, 40, 2), (2, 9, 64, 3)])
def test_linear_brute_force_exact(M, N, K, seed):
    x, W = S.linear_inputs(M, N, K, tag=f"pin{seed}")
    xb, Wb = bf16_bits(x), bf16_bits(W)
    y, a = O.linear_bf16(xb, Wb)
    xf, Wf = bf16_float(xb), bf16_float(Wb)
    ybits = O.round_bf16(y)
    for m in range(M):
        for n in range(N):
            exact = sum((frac(xf[m, k]) * frac(Wf[n, k]) for k in range(K)), Fraction(0))
            absx = sum((abs(frac(xf[m, k]) * frac(Wf[n, k])) for k in range(K)), Fraction(0))
            assert abs(Fraction(y[m, n]) - exact) <= absx * Fraction(1, 2 ** 50)
            assert a[m, n] == pytest.approx(float(absx), rel=1e-14)
            assert int(ybits[m, n]) == bf16_bits_of_exact(exact)


def test_linear_rows_subset_matches_full():
    x, W = S.linear_inputs(2, 33, 48, tag="subset")
    xb, Wb = bf16_bits(x), bf16_bits(W)
    yf, af = O.linear_bf16(xb, Wb)
    rows = np.array([32, 0, 17, 5])
    ys, as_ = O.linear_bf16(xb, Wb, rows=rows)
    assert np.array_equal(ys, yf[:, rows]) and np.array_equal(as_, af[:, rows])


def test_linear_identity_and_one_hot():
    K = 48
    x, W = S.linear_inputs(3, 20, K, tag="onehot")
    xb, Wb = bf16_bits(x), bf16_bits(W)
    eye = bf16_bits(torch.eye(K, dtype=torch.bfloat16))
    y, _ = O.linear_bf16(xb, eye)
    assert np.array_equal(O.round_bf16(y), xb)                 # x . I^T == x
    for k in (0, 13, K - 1):
        e = np.zeros((1, K), np.uint16)
        e[0, k] = 0x3F80                                       # bf16 1.0
        y, _ = O.linear_bf16(e, Wb)
        assert np.array_equal(O.round_bf16(y)[0], Wb[:, k])    # picks column k of W


def test_linear_is_linear_exactly():
    g = torch.Generator().manual_seed(11)
    K, N = 40, 6
    x1 = torch.randint(-8, 9, (1, K), generator=g).to(torch.bfloat16)
    x2 = torch.randint(-8, 9, (1, K), generator=g).to(torch.bfloat16)
    W = torch.randint(-16, 17, (N, K), generator=g).to(torch.bfloat16)
    comb = (2 * x1.float() + x2.float()).to(torch.bfloat16)    # exact: small integers
    Wb = bf16_bits(W)
    y1, _ = O.linear_bf16(bf16_bits(x1), Wb)
    y2, _ = O.linear_bf16(bf16_bits(x2), Wb)
    y3, _ = O.linear_bf16(bf16_bits(comb), Wb)
    assert np.array_equal(y3, 2 * y1 + y2)


def test_linear_against_library_matmul():
    x, W = S.linear_inputs(4, 64, 1024, tag="libmm")
    y, _ = O.linear_bf16(bf16_bits(x), bf16_bits(W))
    ref = (x.double() @ W.double().T).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- SiLU

def test_silu_special_values_and_closed_forms():
    assert O.silu(0.0) == 0.0
    assert O.silu(40.0) == 40.0
    assert O.silu(-800.0) == 0.0 and math.copysign(1, O.silu(-800.0)) < 0
    ln3 = math.log(3.0)
    assert O.silu(ln3) == pytest.approx(0.75 * ln3, rel=1e-15)      # e^-ln3 = 1/3
    for g in (-7.5, -1.25, -0.1, 0.3, 2.0, 9.0):
        assert O.silu(g) - O.silu(-g) == pytest.approx(g, rel=1e-14)  # g*s(g) + g*s(-g) = g
        assert 0.0 < O.silu(g) / g < 1.0
        assert O.silu(g) == pytest.approx(_silu_mp(Fraction(g)), rel=1e-15)


# ---------------------------------------------------------------- gate/up

def test_gate_up_brute_force():
    M, Nh, K = 2, 5, 32
    x, W = S.gate_up_inputs(M, Nh, K)
    xb, Wb = bf16_bits(x), bf16_bits(W)
    res = O.gate_up_silu(xb, Wb)
    xf, Wf = bf16_float(xb), bf16_float(Wb)
    for m in range(M):
        for j in range(Nh):
            g = sum((frac(xf[m, k]) * frac(Wf[2 * j, k]) for k in range(K)), Fraction(0))
            u = sum((frac(xf[m, k]) * frac(Wf[2 * j + 1, k]) for k in range(K)), Fraction(0))
            assert res["g"][m, j] == float(g) and res["u"][m, j] == float(u)
            assert res["out"][m, j] == pytest.approx(_silu_mp(g) * float(u), rel=1e-14, abs=1e-300)


def test_gate_up_interleave_order():
    K, Nh = 16, 3
    Wf = np.zeros((2 * Nh, K))
    for j in range(Nh):
        Wf[2 * j, j] = 1.0          # gate_j = x[j]
        Wf[2 * j + 1, 8 + j] = 1.0  # up_j = x[8+j]
    Wb = bf16_bits(torch.tensor(Wf, dtype=torch.bfloat16))
    x = torch.tensor([[0.5, -2.0, 3.0, 0, 0, 0, 0, 0, 4.0, 0.25, -1.5, 0, 0, 0, 0, 0]],
                     dtype=torch.bfloat16)
    res = O.gate_up_silu(bf16_bits(x), Wb)
    xv = x.double()[0]
    for j in range(Nh):
        expect = float(xv[j]) / (1 + math.exp(-float(xv[j]))) * float(xv[8 + j])
        assert res["out"][0, j] == pytest.approx(expect, rel=1e-15)


def test_gate_up_cols_subset():
    x, W = S.gate_up_inputs(3, 11, 64)
    full = O.gate_up_silu(bf16_bits(x), bf16_bits(W))
    cols = np.array([10, 3, 0])
    sub = O.gate_up_silu(bf16_bits(x), bf16_bits(W), cols=cols)
    for k in full:
        assert np.array_equal(sub[k], full[k][:, cols])


# ---------------------------------------------------------------- fp8 head

def test_head_brute_force_and_one_hot():
    M, N, K = 2, 6, 32
    x, Wq, scale = S.head_inputs(M, N, K)
    xb, Wqn, sc = bf16_bits(x), Wq.numpy(), float(scale[0])
    lg, ab = O.head_fp8(xb, Wqn, sc)
    xf, wf = bf16_float(xb), e4m3_float_lib(Wqn)
    for m in range(M):
        for n in range(N):
            s = sum((frac(xf[m, k]) * frac(wf[n, k]) for k in range(K)), Fraction(0))
            assert lg[m, n] == pytest.approx(float(frac(sc) * s), rel=1e-15, abs=1e-300)
    for k in (0, 31):
        e = np.zeros((1, K), np.uint16)
        e[0, k] = 0x3F80
        lg1, _ = O.head_fp8(e, Wqn, sc)
        assert np.array_equal(lg1[0], sc * wf[:, k])


def test_head_quantised_weights_span_the_e4m3_range():
    _, Wq, scale = S.head_inputs(1, 512, 256)
    vals = e4m3_float_lib(Wq.numpy())
    assert np.nanmax(np.abs(vals)) == 448.0 and not np.isnan(vals).any()


def test_head_argmax_brute_force_ties_and_nan():
    M, N, K = 3, 40, 32
    x, Wq, scale = S.head_inputs(M, N, K)
    xb, Wqn, sc = bf16_bits(x), Wq.numpy().copy(), float(scale[0])
    lg, _ = O.head_fp8(xb, Wqn, sc)
    idx, best, gap = O.head_argmax(xb, Wqn, sc)
    for m in range(M):
        f = lg[m].astype(np.float32)
        assert idx[m] == int(np.argmax(f))          # numpy returns the first maximum
        assert best[m] == f.max()
        assert gap[m] > 0
    # duplicated winning rows: the lowest index wins
    w0 = idx[0]
    Wdup = Wqn.copy()
    Wdup[2] = Wqn[w0]
    Wdup[w0 + 5 if w0 + 5 < N else 0] = Wqn[w0]
    i2, _, _ = O.head_argmax(xb, Wdup, sc)
    assert i2[0] == min(2, w0)
    # all-zero weights: every logit ties at zero -> index 0
    iz, bz, _ = O.head_argmax(xb, np.zeros_like(Wqn), sc)
    assert list(iz) == [0] * M and list(bz) == [0.0] * M
    # a NaN code row is never picked
    Wn = Wqn.copy()
    Wn[w0, 0] = 0x7F
    i3, _, _ = O.head_argmax(xb, Wn, sc)
    assert i3[0] != w0


# ---------------------------------------------------------------- MoE

def _route_brute(ids, E):
    M, topk = ids.shape
    valid = np.zeros_like(ids)
    for t in range(M):
        seen = set()
        for k in range(topk):
            e = int(ids[t, k])
            if 0 <= e < E and e not in seen:
                valid[t, k] = 1
            seen.add(e)
    groups = {}
    for t in range(M):
        for k in range(topk):
            if valid[t, k]:
                groups.setdefault(int(ids[t, k]), []).append((t, k))
    return valid, groups


@pytest.mark.parametrize("M", [1, 2, 5, 16])
def test_moe_route_brute_force(M):
    ids, _ = S.moe_routing(M, 6, 128, seed=100 + M)
    ids = ids.numpy()
    r = O.moe_route(ids, 128)
    valid, groups = _route_brute(ids, 128)
    assert np.array_equal(r["valid"], valid)
    assert list(r["experts"]) == sorted(groups)
    for u, e in enumerate(r["experts"]):
        lo, hi = r["offsets"][u], r["offsets"][u + 1]
        assert list(zip(r["pair_tok"][lo:hi], r["pair_slot"][lo:hi])) == groups[e]


def test_moe_route_invalid_ids():
    ids = np.array([[3, 3, 200, -1, 7, 3], [0, 1, 2, 3, 4, 5]], np.int32)
    r = O.moe_route(ids, 8)
    assert r["valid"].tolist() == [[1, 0, 0, 0, 1, 0], [1, 1, 1, 1, 1, 1]]
    assert list(r["experts"]) == [0, 1, 2, 3, 4, 5, 7]


def _tiny_moe(M=2, topk=3, E=5, I=4, K=32, Nout=6):
    W1q, s1, W2q, s2 = S.moe_weights(E, I, K, Nout)
    x, ids, gw = S.moe_inputs(M, K, topk, E)
    return x, ids, gw, W1q, s1, W2q, s2


def test_moe_w1_brute_force():
    x, ids, gw, W1q, s1, W2q, s2 = _tiny_moe()
    xb = bf16_bits(x)
    res = O.moe_w1_silu(xb, ids.numpy(), W1q.numpy(), s1.numpy())
    xf = bf16_float(xb)
    w1 = e4m3_float_lib(W1q.numpy())
    s1n = s1.numpy().astype(np.float64)
    M, topk = ids.shape
    I = W1q.shape[1] // 2
    for t in range(M):
        for k in range(topk):
            e = int(ids[t, k])
            for j in range(I):
                g = frac(s1n[e, j]) * sum((frac(xf[t, q]) * frac(w1[e, j, q]) for q in range(xf.shape[1])), Fraction(0))
                u = frac(s1n[e, I + j]) * sum((frac(xf[t, q]) * frac(w1[e, I + j, q]) for q in range(xf.shape[1])), Fraction(0))
                assert res["g"][t, k, j] == pytest.approx(float(g), rel=1e-15, abs=1e-300)
                assert res["u"][t, k, j] == pytest.approx(float(u), rel=1e-15, abs=1e-300)
                assert res["a"][t, k, j] == pytest.approx(_silu_mp(g) * float(u), rel=1e-14, abs=1e-300)


def test_moe_w1_invalid_slot_is_zero():
    x, ids, gw, W1q, s1, W2q, s2 = _tiny_moe()
    bad = ids.numpy().copy()
    bad[0, 1] = bad[0, 0]
    bad[1, 2] = 99
    res = O.moe_w1_silu(bf16_bits(x), bad, W1q.numpy(), s1.numpy())
    assert not res["a"][0, 1].any() and not res["a"][1, 2].any()
    assert res["a"][0, 0].any()


def test_moe_w2_brute_force_and_reductions():
    x, ids, gw, W1q, s1, W2q, s2 = _tiny_moe()
    M, topk = ids.shape
    E, Nout, I = W2q.shape
    g = torch.Generator().manual_seed(5)
    a = torch.randn((M, topk, I), generator=g).to(torch.bfloat16)
    ab = bf16_bits(a)
    y, bound = O.moe_w2(ab, ids.numpy(), gw.numpy(), W2q.numpy(), s2.numpy())
    af = bf16_float(ab)
    w2 = e4m3_float_lib(W2q.numpy())
    gwn, s2n = gw.numpy(), s2.numpy()
    for t in range(M):
        for n in range(Nout):
            tot = Fraction(0)
            for k in range(topk):
                e = int(ids[t, k])
                h = sum((frac(af[t, k, i]) * frac(w2[e, n, i]) for i in range(I)), Fraction(0))
                tot += frac(gwn[t, k]) * frac(s2n[e, n]) * h
            assert y[t, n] == pytest.approx(float(tot), rel=1e-14, abs=1e-300)
    # one token, one slot, gate weight 1: a per-row-scaled fp8 GEMV of a
    ids1 = ids.numpy()[:1, :1]
    y1, _ = O.moe_w2(ab[:1, :1], ids1, np.ones((1, 1), np.float32), W2q.numpy(), s2.numpy())
    e = int(ids1[0, 0])
    ref = (af[0, 0] @ w2[e].T) * s2n[e]
    assert np.allclose(y1[0], ref, rtol=1e-13, atol=1e-300)
    # every slot on identical experts with equal gate weights = that expert's result
    W2same = np.broadcast_to(W2q.numpy()[:1], W2q.shape).copy()
    s2same = np.broadcast_to(s2n[:1], s2n.shape).copy()
    a_same = np.broadcast_to(ab[:, :1], ab.shape).copy()
    gw_eq = np.full((M, topk), 1.0 / 4, np.float32)
    ys, _ = O.moe_w2(a_same, ids.numpy(), gw_eq, W2same, s2same)
    single = np.stack([(af[t, 0] @ w2[0].T) * s2n[0] for t in range(M)])
    assert np.allclose(ys, single * topk / 4, rtol=1e-13)


# ---------------------------------------------------------------- A8W8 blockscale

def _e4m3_encode_lib(v32: np.ndarray) -> np.ndarray:
    """binary32 values -> e4m3 codes by torch's own float8_e4m3fn cast (round to nearest
    even), after clamping to +-448 (the saturating conversion)."""
    t = torch.from_numpy(np.asarray(v32, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_hand_worked_points():
    with open(os.path.join(GOLDEN, "e4m3_rne_points.txt")) as f:
        rows = [ln.split()[:2] for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 12
    for val, code in rows:
        assert O.e4m3_encode(float(Fraction(val))) == int(code, 16), (val, code)


def test_e4m3_encode_matches_library_rounding():
    finite = [c for c in range(0x7F)]
    vals = [O.e4m3_value(c) for c in finite]
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]                 # exact ties
    g = np.random.default_rng(11)
    rnd = (g.standard_normal(20000) * np.exp2(g.uniform(-12, 10, 20000))).astype(np.float32)
    pts = np.concatenate([np.float32(vals), np.float32(mids), np.nextafter(np.float32(mids), np.float32(0)),
                          np.nextafter(np.float32(mids), np.float32(1e9)), rnd, -rnd[:2000]]).astype(np.float32)
    lib = _e4m3_encode_lib(pts)
    got = np.array([O.e4m3_encode(float(v)) for v in pts], np.uint8)
    assert np.array_equal(got, lib), pts[got != lib][:8]
    # every finite code round-trips
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert O.e4m3_encode(O.e4m3_value(c)) == (c if c != 0x80 else 0x80), hex(c)


def _quant_numpy(xbits: np.ndarray):
    """Per (token, 128-block) quantisation written with numpy binary32 arithmetic and
    torch's e4m3 cast (independent of the oracle's C code)."""
    x = bf16_float(xbits).astype(np.float32)
    M, K = x.shape
    nb = (K + 127) // 128
    q = np.zeros((M, K), np.uint8)
    sx = np.zeros((M, nb), np.float32)
    for m in range(M):
        for b in range(nb):
            blk = x[m, b * 128:(b + 1) * 128]
            amax = np.float32(np.max(np.abs(blk)))
            amax = max(amax, np.float32(2.0 ** -32))
            r = np.float32(448.0) / amax
            sx[m, b] = amax / np.float32(448.0)
            q[m, b * 128:(b + 1) * 128] = _e4m3_encode_lib(blk * r)
    return q, sx


def _a8_inputs(M, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((M, K), generator=g)
    nb = (K + 127) // 128
    x *= torch.exp2(torch.randint(-20, 12, (M, nb), generator=g).float()).repeat_interleave(128, 1)[:, :K]
    x[0, 128:256] = 0.0                                  # an all-zero block
    if K > 300:
        x[-1, 300] = 3.0e4                               # a spike that owns its block's scale
    return bf16_bits(x.to(torch.bfloat16))


@pytest.mark.parametrize("M,K,seed", [(3, 272, 1), (2, 1040, 2), (5, 128, 3)])
def test_a8_quant_matches_independent_binary32(M, K, seed):
    xb = _a8_inputs(M, K, seed)
    q, sx = O.a8_quant(xb)
    q_ref, sx_ref = _quant_numpy(xb)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(sx.view(np.uint32), sx_ref.view(np.uint32))
    if K >= 256:
        assert (q[0, 128:256] == 0).all() and sx[0, 1] == np.float32(2.0 ** -32) / np.float32(448.0)
    # every block that is not all zero has its largest magnitude on the top code, 448
    qv = np.abs(e4m3_float_lib(q))
    for m in range(M):
        for b in range((K + 127) // 128):
            blk = qv[m, b * 128:(b + 1) * 128]
            assert blk.max() in (0.0, 448.0), (m, b, blk.max())


def _a8w8_exact(q, sx, Wq, sw, K):
    M, N = q.shape[0], Wq.shape[0]
    nb = (K + 127) // 128
    qv = e4m3_float_lib(q)
    wv = e4m3_float_lib(Wq)
    y = np.empty((M, N), object)
    ad = np.empty((M, N), object)
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            a = Fraction(0)
            for b in range(nb):
                c = frac(sx[m, b]) * frac(sw[n // 128, b])
                d = sum((frac(qv[m, k]) * frac(wv[n, k]) for k in range(b * 128, min(K, b * 128 + 128))), Fraction(0))
                da = sum((abs(frac(qv[m, k]) * frac(wv[n, k])) for k in range(b * 128, min(K, b * 128 + 128))),
                         Fraction(0))
                s += c * d
                a += abs(c) * da
            y[m, n] = s
            ad[m, n] = a
    return y, ad


def _a8w8_weights(N, K, seed):
    g = torch.Generator().manual_seed(seed)
    Wq = (torch.randn((N, K), generator=g) * 60).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    nbn, nbk = (N + 127) // 128, (K + 127) // 128
    sw = (torch.rand((nbn, nbk), generator=g) * 1e-3 + 1e-4).numpy().astype(np.float32)
    return Wq, sw


def test_a8w8_linear_brute_force_exact():
    """N = 130 puts rows 128..129 in the second weight-scale row; K = 272 makes three
    K-blocks, the last one short: a wrong block index or a transposed scale fails."""
    M, N, K = 2, 130, 272
    xb = _a8_inputs(M, K, 5)
    q, sx = O.a8_quant(xb)
    Wq, sw = _a8w8_weights(N, K, 6)
    rows = np.array([0, 1, 63, 127, 128, 129])
    y, ad = O.a8w8_linear_q(q, sx, Wq, sw, rows=rows)
    # exact sums, each row with its own weight-scale row n // 128
    ye = np.empty((M, len(rows)), object)
    ae = np.empty((M, len(rows)), object)
    for j, n in enumerate(rows):
        sw_row = np.zeros_like(sw)
        sw_row[0] = sw[n // 128]
        yy, aa = _a8w8_exact(q, sx, Wq[n:n + 1], sw_row, K)
        ye[:, j], ae[:, j] = yy[:, 0], aa[:, 0]
    for m in range(M):
        for j in range(len(rows)):
            tol = 1e-13 * float(ae[m, j]) + 1e-300
            assert abs(y[m, j] - float(ye[m, j])) <= tol, (m, j)
            assert abs(ad[m, j] - float(ae[m, j])) <= tol


def test_a8w8_one_hot_closed_form():
    """x = v e_k: the token's block holds one nonzero, which quantises to +-448, so
    y[n] = sx * sw[n/128, k/128] * 448 * e4m3(W[n, k]) * sign(v)."""
    M, N, K = 1, 260, 384
    Wq, sw = _a8w8_weights(N, K, 8)
    for k, v in [(5, 3.25), (200, -0.0078125), (383, 1.5e3)]:
        x = torch.zeros((M, K))
        x[0, k] = v
        xb = bf16_bits(x.to(torch.bfloat16))
        r = O.a8w8_linear(xb, Wq, sw)
        q = r["q"]
        assert q[0, k] == (0x7E if v > 0 else 0xFE) and np.count_nonzero(q) == 1
        amax = np.float32(abs(np.float32(bf16_float(xb)[0, k])))
        sxv = float(amax / np.float32(448.0))
        assert r["sx"][0, k // 128] == np.float32(sxv)
        w = e4m3_float_lib(Wq[:, k])
        want = sxv * sw[np.arange(N) // 128, k // 128].astype(np.float64) * 448.0 * w * np.sign(v)
        assert np.allclose(r["y"][0], want, rtol=1e-15, atol=0)


def test_a8w8_reduces_to_head_when_scales_are_one():
    """Blocks whose largest magnitude is exactly 448 and whose values are e4m3 numbers
    quantise to themselves with sx = 1; with one weight scale c everywhere the step is
    the fp8 head with scale c."""
    M, N, K = 3, 140, 384
    g = torch.Generator().manual_seed(9)
    xv = (torch.randn((M, K), generator=g) * 50).clamp(-440, 440).to(torch.float8_e4m3fn).to(torch.float32)
    xv[:, ::128] = 448.0                                 # every block's max is 448
    xb = bf16_bits(xv.to(torch.bfloat16))
    Wq, _ = _a8w8_weights(N, K, 10)
    c = np.float32(0.0078125)
    sw = np.full(((N + 127) // 128, K // 128), c, np.float32)
    r = O.a8w8_linear(xb, Wq, sw)
    assert (r["sx"] == 1.0).all()
    assert np.array_equal(e4m3_float_lib(r["q"]), bf16_float(xb))
    lg, ad = O.head_fp8(xb, Wq, float(c))
    assert np.allclose(r["y"], lg, rtol=1e-14, atol=1e-300)
    assert np.allclose(r["absdot"], ad, rtol=1e-14, atol=1e-300)


def test_a8w8_weight_scale_is_linear_exactly():
    M, N, K = 2, 200, 256
    xb = _a8_inputs(M, K, 12)
    Wq, sw = _a8w8_weights(N, K, 13)
    y1 = O.a8w8_linear(xb, Wq, sw)["y"]
    y2 = O.a8w8_linear(xb, Wq, (sw * np.float32(2.0)).astype(np.float32))["y"]
    assert np.array_equal(y2, 2.0 * y1)


def test_a8_quant_non_finite_reading():
    """Reading of the pages' silence on non-finite activations: an inf in a block makes
    that block's scale inf and its codes NaN/zero, so the token's outputs are NaN; the
    other tokens are untouched.  Saturation maps +-inf inputs of the encoder to +-448."""
    assert O.e4m3_encode(float("inf")) == 0x7E and O.e4m3_encode(float("-inf")) == 0xFE
    M, N, K = 2, 130, 256
    x = torch.ones((M, K))
    x[0, 3] = float("inf")
    xb = bf16_bits(x.to(torch.bfloat16))
    Wq, sw = _a8w8_weights(N, K, 14)
    r = O.a8w8_linear(xb, Wq, sw)
    assert np.isinf(r["sx"][0, 0]) and np.isfinite(r["sx"][1]).all()
    assert np.isnan(r["y"][0]).all() and np.isfinite(r["y"][1]).all()
