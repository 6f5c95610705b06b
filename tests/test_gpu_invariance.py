"""Batch-invariant numerics mode: output row m is a function of input row m alone.

With DG_NUMERICS_BATCH_INVARIANT every row bucket of an op runs one kernel family
with one reduction order fixed by the shape, so a row computed inside a call of M
rows has the same bits as the same row computed alone, for every M the op takes,
and permuting the rows permutes the outputs.  The rows still meet the oracle's
bounds (checked on rows computed alone, where the fastest mode would have taken
the CUDA cores).
"""
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import oracle as O
from oracle import tolerance as T
from synth import decode_inputs as S
from tests._helpers import bits16, f64, sample_rows, lin_excess, silu_excess

pytestmark = pytest.mark.gpu

LIN_M = [1, 2, 3, 4, 5, 8, 13, 16, 17, 32, 33, 64, 100, 128, 129, 192, 256, 257, 384, 512]


@pytest.fixture(autouse=True)
def invariant_mode():
    dg.dg_set_numerics(dg.DG_NUMERICS_BATCH_INVARIANT)
    yield
    dg.dg_set_numerics(dg.DG_NUMERICS_FASTEST)


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


def _perm(n, seed, device):
    return torch.randperm(n, generator=torch.Generator().manual_seed(seed)).to(device)


@pytest.mark.parametrize("N,K", [(4096, 4096), (257, 1096), (2048, 1024), (12288, 4096), (32768, 1024)])
def test_linear_rows_independent_of_the_batch(cuda_device, N, K):
    x, W = S.linear_inputs(512, N, K, device=cuda_device)
    full = dg.dg_gemv_bf16(x, W)
    for M in LIN_M:
        assert _same(dg.dg_gemv_bf16(x[:M].contiguous(), W), full[:M]), M
    p = _perm(512, N + K, cuda_device)
    assert _same(dg.dg_gemv_bf16(x[p].contiguous(), W), full[p])
    # one row alone (the fastest mode's CUDA-core bucket) against the fp64 oracle
    cols = sample_rows(N, 128, seed=N ^ K)
    ci = torch.as_tensor(cols, device=cuda_device)
    ref, ad = O.linear_bf16(bits16(x[:1]), bits16(W[ci]))
    y1 = dg.dg_gemv_bf16(x[:1].contiguous(), W)
    assert (lin_excess(f64(y1[:, ci]), ref, ad) <= 0).all()


@pytest.mark.parametrize("Nh,K", [(700, 4096), (12288, 4096), (96, 1544)])
def test_gate_up_rows_independent_of_the_batch(cuda_device, Nh, K):
    x, Wgu = S.gate_up_inputs(512, Nh, K, device=cuda_device)
    full = dg.dg_gate_up_silu(x, Wgu)
    for M in LIN_M:
        assert _same(dg.dg_gate_up_silu(x[:M].contiguous(), Wgu), full[:M]), M
    p = _perm(512, Nh + K, cuda_device)
    assert _same(dg.dg_gate_up_silu(x[p].contiguous(), Wgu), full[p])
    c = torch.as_tensor(sample_rows(Nh, 48, seed=Nh), device=cuda_device)
    rows = torch.stack((2 * c, 2 * c + 1), dim=1).reshape(-1)
    r = O.gate_up_silu(bits16(x[:1]), bits16(Wgu[rows]))
    out1 = dg.dg_gate_up_silu(x[:1].contiguous(), Wgu)
    exc = silu_excess(f64(out1[:, c]), r["g"], r["u"], r["absg"], r["absu"], r["out"])
    assert (exc <= 0).all()


# (N, K, most rows): K = 16384 stays on the CUDA cores, which stage all rows' activations
@pytest.mark.parametrize("N,K,top", [(20000, 4096, 8), (3000, 16384, 3)])
def test_head_rows_and_picks_independent_of_the_batch(cuda_device, N, K, top):
    x, Wq, scale = S.head_inputs(top, N, K, device=cuda_device)
    lg8, am8 = dg.dg_head_fp8_argmax(x, Wq, scale)
    for M in range(1, top):
        lg, am = dg.dg_head_fp8_argmax(x[:M].contiguous(), Wq, scale)
        assert _same(lg, lg8[:M]) and torch.equal(am, am8[:M]), M
    p = _perm(top, N, cuda_device)
    lg, am = dg.dg_head_fp8_argmax(x[p].contiguous(), Wq, scale)
    assert _same(lg, lg8[p]) and torch.equal(am, am8[p])
    rows = sample_rows(N, 64, seed=N)
    ri = torch.as_tensor(rows, device=cuda_device)
    ref, ad = O.head_fp8(bits16(x[:1]), Wq[ri].cpu().numpy(), float(scale.cpu()[0]))
    assert (lin_excess(f64(lg8[:1, ri]), ref, ad) <= 0).all()


@pytest.mark.parametrize("E,I,K,Nout", [(128, 1536, 4096, 4096), (24, 192, 528, 200)])
def test_moe_tokens_independent_of_the_batch(cuda_device, E, I, K, Nout):
    W1q, s1, W2q, s2 = S.moe_weights(E, I, K, Nout, device=cuda_device)
    x, ids, gw = S.moe_inputs(16, K, 6, E, device=cuda_device)
    a16 = dg.dg_moe_w1_silu(x, ids, W1q, s1)
    y16 = dg.dg_moe_w2(a16, ids, gw, W2q, s2)
    for M in range(1, 16):
        a = dg.dg_moe_w1_silu(x[:M].contiguous(), ids[:M].contiguous(), W1q, s1)
        assert _same(a, a16[:M]), M
        y = dg.dg_moe_w2(a16[:M].contiguous(), ids[:M].contiguous(), gw[:M].contiguous(), W2q, s2)
        assert _same(y, y16[:M]), M
    p = _perm(16, E + I, cuda_device)
    a = dg.dg_moe_w1_silu(x[p].contiguous(), ids[p].contiguous(), W1q, s1)
    assert _same(a, a16[p])
    y = dg.dg_moe_w2(a16[p].contiguous(), ids[p].contiguous(), gw[p].contiguous(), W2q, s2)
    assert _same(y, y16[p])
    # a token alone, with the other 15 tokens replaced by different routings
    x2, ids2, gw2 = S.moe_inputs(16, K, 6, E, rep=1, device=cuda_device)
    x2[3], ids2[3], gw2[3] = x[3], ids[3], gw[3]
    a2 = dg.dg_moe_w1_silu(x2, ids2, W1q, s1)
    assert _same(a2[3], a16[3])
    a2[3] = a16[3]
    assert _same(dg.dg_moe_w2(a2, ids2, gw2, W2q, s2)[3], y16[3])
