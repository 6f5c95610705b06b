"""Position-complete exactness checks on the GPU, where the tolerance is blind.

The stated bound (4e-3 * sum|x*w| + 1e-5) is wide enough that a kernel dropping or
double-counting a few dozen k-terms of a long row could pass it.  These checks have
exact answers instead, at the K lengths where the K-split ranks, the cluster fold and
the short last segment engage:
  * W = I: y == x bit for bit (one product per output, the fold adds zeros);
  * one-hot x = e_k: y[n] == W[n, k] (bf16 linear) and logit[n] ==
    bf16_rn(fp32(e4m3(Wq[n, k])) * scale) with the pick on those fp32 values (fp8 head);
  * MoE x -> W1 -> W2 -> y end to end against the fp64 chain, with the W1 error bound
    propagated through W2.
"""
import numpy as np
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import oracle as O
from oracle import tolerance as T
from synth import decode_inputs as S
from tests._helpers import bits16, f64, lin_excess

pytestmark = pytest.mark.gpu

CCW = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0)
CCW_KS = dg.Choice.make(dg.DG_VAR_CC_WARP, 2, 8, 0, 4)      # four warps share a row group's segments
BULK = dg.Choice.make(dg.DG_VAR_CC_BULK, 0, 0, 0)
TC = dg.Choice.make(dg.DG_VAR_TC, 0)
MMA = dg.Choice.make(dg.DG_VAR_MMA, 0, 0, 0, 0)
LIN_CASES = [("cc", CCW, 1), ("cc_ksplit", CCW_KS, 2), ("bulk", BULK, 1), ("cc", CCW, 5),
             ("tc", TC, 3), ("tc", TC, 16), ("tc", TC, 128), ("default", None, 8),
             ("mma", MMA, 3), ("mma", MMA, 12), ("mma", MMA, 16)]
LONG_K = [4096, 12288, 4096 + 16]


def _one_hot_positions(K):
    """Segment edges, the last element, and the first and last of the short tail."""
    ks = {0, 1, 511, 512, 1023, 1024, 2047, 4095, K - 16, K - 1}
    return sorted(k for k in ks if 0 <= k < K)


@pytest.fixture(scope="module")
def eyes(cuda_device):
    return {K: torch.eye(K, dtype=torch.bfloat16, device=cuda_device) for K in LONG_K}


@pytest.mark.parametrize("K", LONG_K)
@pytest.mark.parametrize("name,choice,M", LIN_CASES, ids=[f"{n}-M{m}" for n, _, m in LIN_CASES])
def test_linear_identity_exact_long_k(cuda_device, eyes, K, name, choice, M):
    x, _ = S.linear_inputs(M, 8, K, device=cuda_device, tag="exact")
    y = dg.dg_gemv_bf16(x, eyes[K], choice=choice)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))


@pytest.mark.parametrize("K", LONG_K)
@pytest.mark.parametrize("name,choice,M", LIN_CASES, ids=[f"{n}-M{m}" for n, _, m in LIN_CASES])
def test_linear_one_hot_exact_long_k(cuda_device, K, name, choice, M):
    N = 1000
    _, W = S.linear_inputs(1, N, K, device=cuda_device, tag="exact")
    pos = _one_hot_positions(K)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=cuda_device)
    ks = [pos[m % len(pos)] for m in range(M)]
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    y = dg.dg_gemv_bf16(x, W, choice=choice)
    torch.cuda.synchronize()
    want = W[:, ks].t().contiguous()
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def _head_one_hot_want(Wq, scale, ks):
    """logit[m, n] = fp32(e4m3(Wq[n, k_m]) * scale) (one fp32 multiply, round to nearest
    even), its bf16 rounding, and the lowest index of the largest fp32 logit."""
    dec = Wq[:, ks].cpu().view(torch.float8_e4m3fn).to(torch.float32).t().contiguous()    # [M, N]
    logit = dec * scale.cpu()[0]
    return logit.to(torch.bfloat16), torch.argmax(logit, dim=1).to(torch.int32)


@pytest.mark.parametrize("K", [4096, 4096 + 16])
@pytest.mark.parametrize("family,M", [("cc", 1), ("cc", 3), ("cc", 8), ("bulk", 2), ("tc", 2), ("tc", 5),
                                      ("tc", 8), ("default", 1), ("default", 4)])
def test_head_one_hot_exact(cuda_device, K, family, M):
    choice = {"cc": CCW, "bulk": BULK, "tc": TC, "default": None}[family]
    N = 5000
    _, Wq, scale = S.head_inputs(1, N, K, device=cuda_device)
    pos = _one_hot_positions(K)
    ks = [pos[(3 * m + 1) % len(pos)] for m in range(M)]
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=cuda_device)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    logits, am = dg.dg_head_fp8_argmax(x, Wq, scale, choice=choice)
    torch.cuda.synchronize()
    want_l, want_am = _head_one_hot_want(Wq, scale, ks)
    # equal as values (a zero code may be +0 or -0; the chain's sum of zero products
    # carries no sign rule), otherwise bit for bit
    assert torch.equal(logits.cpu().float(), want_l.float())
    assert torch.equal(am.cpu(), want_am)      # torch.argmax returns the first of equal maxima


# ---------------------------------------------------------------- MoE end to end

E, I, KH, TOPK = 128, 1536, 4096, 6


@pytest.fixture(scope="module")
def moe_w(cuda_device):
    return S.moe_weights(E, I, KH, KH, device=cuda_device)


def _dec(codes_u8):
    return torch.from_numpy(np.ascontiguousarray(codes_u8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("family", ["default", "cc", "tc", "range"])
@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_moe_end_to_end_against_oracle(cuda_device, moe_w, M, family):
    """y = W2(silu(W1 x)) through both kernels, against the fp64 chain on the oracle's
    own activations: |y - y_ref| <= W2's bound on the GPU's a + sum_k |gw| s2 |W2| err_a,
    err_a being W1's bound for each element of a."""
    choice = {"default": None, "cc": dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0, 0, 2), "tc": TC,
              "range": dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0, 0, 2, 2)}[family]
    W1q, s1, W2q, s2 = moe_w
    x, ids, gw = S.moe_inputs(M, KH, TOPK, E, rep=5, device=cuda_device)
    a = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=choice)
    y = dg.dg_moe_w2(a, ids, gw, W2q, s2, choice=choice)
    torch.cuda.synchronize()
    ids_np = ids.cpu().numpy()
    used = np.unique(ids_np)
    remap = {int(e): i for i, e in enumerate(used)}
    ids_c = np.vectorize(lambda e: remap[int(e)])(ids_np).astype(np.int32)
    sel = torch.as_tensor(used, device=cuda_device)
    w1c, s1c = W1q[sel].cpu().numpy(), s1[sel].cpu().numpy()
    w2c, s2c = W2q[sel].cpu().numpy(), s2[sel].cpu().numpy().astype(np.float64)
    r1 = O.moe_w1_silu(bits16(x), ids_c, w1c, s1c)
    err_a = T.silu_mul_bound(r1["g"], r1["u"], r1["absg"], r1["absu"], r1["a"])     # [M, topk, I]
    _, b2 = O.moe_w2(bits16(a), ids_c, gw.cpu().numpy(), w2c, s2c.astype(np.float32))
    gwn = gw.cpu().numpy().astype(np.float64)
    y_ref = np.zeros((M, KH))
    prop = np.zeros((M, KH))
    for u in range(len(used)):
        w2 = _dec(w2c[u])                                  # [Nout, I]
        for t in range(M):
            for k in range(TOPK):
                if ids_c[t, k] != u:
                    continue
                y_ref[t] += gwn[t, k] * (s2c[u] * (w2 @ r1["a"][t, k]))
                prop[t] += abs(gwn[t, k]) * (s2c[u] * (np.abs(w2) @ err_a[t, k]))
    err = np.abs(f64(y) - y_ref)
    bound = T.REL * b2 + T.ABS + prop
    exc = lin_excess(f64(y), y_ref, (b2 + prop / T.REL))
    assert (err <= bound).all() and (exc <= 0).all(), f"max err/bound {np.max(err / bound):.3f}"
