"""GPU parity of the fp8-e4m3 vocabulary head and its fused greedy argmax."""
import numpy as np
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import oracle as O
from oracle import tolerance as T
from synth import decode_inputs as S
from tests._helpers import bits16, f64, sample_rows, lin_excess, silu_excess

pytestmark = pytest.mark.gpu

HEAD_M = [1, 2, 3, 4, 8]


def _check_logits(x, Wq, scale, logits, rows=None):
    sc = float(scale.cpu()[0])
    Wn = (Wq if rows is None else Wq[torch.as_tensor(rows, device=Wq.device)]).cpu().numpy()
    lg, ad = O.head_fp8(bits16(x), Wn, sc)
    got = f64(logits if rows is None else logits[:, torch.as_tensor(rows, device=logits.device)])
    exc = lin_excess(got, lg, ad)
    assert (exc <= 0).all(), f"max excess {exc.max():.3e}"


def _check_argmax(x, Wq, scale, am):
    """Exact index unless the oracle's top-2 gap is within twice the error bound (then any
    index whose exact logit is within that window of the maximum is accepted)."""
    sc = float(scale.cpu()[0])
    xb, Wn = bits16(x), Wq.cpu().numpy()
    idx, best, gap = O.head_argmax(xb, Wn, sc)
    got = am.cpu().numpy()
    for m in range(x.shape[0]):
        if got[m] == idx[m]:
            continue
        lg, ad = O.head_fp8(xb[m:m + 1], Wn, sc, rows=np.array([idx[m], got[m]]))
        window = 2 * (T.REL * ad[0].max() + T.ABS)
        assert gap[m] <= window and lg[0, 0] - lg[0, 1] <= window, (m, got[m], idx[m], gap[m])


FAMILIES = {"default": None, "cc": dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0),
            "bulk": dg.Choice.make(dg.DG_VAR_CC_BULK, 0, 0, 0), "tc": dg.Choice.make(dg.DG_VAR_TC, 0)}


@pytest.mark.parametrize("family", ["default", "cc", "bulk", "tc"])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 4096), (2, 777, 1040), (3, 4099, 512), (5, 300, 2064),
                                   (8, 2048, 4096), (4, 1, 16), (6, 130, 4096)])
def test_head_small_exhaustive(cuda_device, M, N, K, family):
    x, Wq, scale = S.head_inputs(M, N, K, device=cuda_device)
    c = FAMILIES[family]
    logits, am = dg.dg_head_fp8_argmax(x, Wq, scale, choice=c)
    torch.cuda.synchronize()
    _check_logits(x, Wq, scale, logits)
    _check_argmax(x, Wq, scale, am)


@pytest.fixture(scope="module")
def full_head(cuda_device):
    x8, Wq, scale = S.head_inputs(8, 248320, 4096, device=cuda_device)
    return x8, Wq, scale


@pytest.mark.parametrize("M", HEAD_M)
def test_head_full_size(cuda_device, full_head, M):
    x8, Wq, scale = full_head
    x = x8[:M].contiguous()
    logits, am = dg.dg_head_fp8_argmax(x, Wq, scale)
    torch.cuda.synchronize()
    _check_logits(x, Wq, scale, logits, rows=sample_rows(248320, 128, seed=M))
    _check_argmax(x, Wq, scale, am)
    # the argmax-only call (no logits buffer) picks the same indices
    _, am2 = dg.dg_head_fp8_argmax(x, Wq, scale, want_logits=False)
    assert torch.equal(am, am2)


def test_head_tc_variants_bitwise_identical(cuda_device):
    x, Wq, scale = S.head_inputs(6, 20000, 4096, device=cuda_device)
    ref_l, ref_a = dg.dg_head_fp8_argmax(x, Wq, scale, choice=FAMILIES["tc"])
    for st in (2, 3, 5, 8):
        l, a = dg.dg_head_fp8_argmax(x, Wq, scale, choice=dg.Choice.make(dg.DG_VAR_TC, st))
        assert torch.equal(l.view(torch.int16), ref_l.view(torch.int16)), st
        assert torch.equal(a, ref_a), st
    for _ in range(3):
        l, a = dg.dg_head_fp8_argmax(x, Wq, scale, choice=FAMILIES["tc"])
        assert torch.equal(l.view(torch.int16), ref_l.view(torch.int16)) and torch.equal(a, ref_a)


def test_head_tc_activations_with_wide_dynamic_range(cuda_device):
    """The hi/lo e4m3 split of the activations: tiny and large entries in one row."""
    M, N, K = 3, 3000, 2048
    x, Wq, scale = S.head_inputs(M, N, K, device=cuda_device)
    g = torch.Generator().manual_seed(9)
    mag = torch.exp2(torch.randint(-30, 12, (M, K), generator=g).float())
    x = (torch.randn((M, K), generator=g) * mag).to(torch.bfloat16).to(cuda_device)
    logits, am = dg.dg_head_fp8_argmax(x, Wq, scale, choice=FAMILIES["tc"])
    torch.cuda.synchronize()
    _check_logits(x, Wq, scale, logits)
    _check_argmax(x, Wq, scale, am)


@pytest.mark.parametrize("M", [1, 5])
def test_head_variants_bitwise_identical(cuda_device, M):
    x, Wq, scale = S.head_inputs(M, 3001, 2064, device=cuda_device)
    ref_l, ref_a = dg.dg_head_fp8_argmax(x, Wq, scale, choice=FAMILIES["cc"])
    choices = [dg.Choice.make(dg.DG_VAR_CC_WARP, R, wpc, cap, ks)
               for R in (1, 2, 4, 8) for wpc in (2, 4, 8) for cap in (0, 1) for ks in (0, 2)]
    choices += [dg.Choice.make(dg.DG_VAR_CC_BULK, 0, st, cps) for st in (0, 2, 5, 16) for cps in (1, 2)]
    for c in choices:
        try:
            l, a = dg.dg_head_fp8_argmax(x, Wq, scale, choice=c)
        except dg.DGError as e:            # a depth that does not fit shared memory for this shape
            assert e.status in (3, 8) and c.variant == dg.DG_VAR_CC_BULK, (repr(c), e.status)
            continue
        assert torch.equal(l.view(torch.int16), ref_l.view(torch.int16)), repr(c)
        assert torch.equal(a, ref_a), repr(c)


@pytest.mark.parametrize("family", ["cc", "bulk", "tc"])
def test_head_ties_go_to_lowest_index(cuda_device, family):
    M, N, K = 3, 5000, 1024
    c = FAMILIES[family]
    x, Wq, scale = S.head_inputs(M, N, K, device=cuda_device)
    _, am = dg.dg_head_fp8_argmax(x, Wq, scale, choice=c)
    for m in range(M):
        w = int(am[m])
        p = (w + 1234) % N                    # a later (or wrapped, earlier) copy of the winner row
        W2 = Wq.clone()
        W2[p] = Wq[w]
        _, am2 = dg.dg_head_fp8_argmax(x[m:m + 1].contiguous(), W2, scale, choice=c)
        assert int(am2[0]) == min(w, p), (m, w, p, int(am2[0]))
    zeros = torch.zeros_like(Wq)
    l0, a0 = dg.dg_head_fp8_argmax(x, zeros, scale, choice=c)
    assert a0.tolist() == [0] * M and (l0.float() == 0).all()


@pytest.mark.parametrize("family", ["cc", "tc"])
def test_head_nan_rows_never_win(cuda_device, family):
    M, N, K = 2, 600, 512
    c = FAMILIES[family]
    x, Wq, scale = S.head_inputs(M, N, K, device=cuda_device)
    _, am = dg.dg_head_fp8_argmax(x, Wq, scale, choice=c)
    W2 = Wq.clone()
    for m in range(M):
        W2[int(am[m]), 7] = 0x7F             # e4m3 NaN code
    _, am2 = dg.dg_head_fp8_argmax(x, W2, scale, choice=c)
    idx, _, _ = O.head_argmax(bits16(x), W2.cpu().numpy(), float(scale.cpu()[0]))
    assert am2.cpu().numpy().tolist() == idx.tolist()
    allnan = torch.full_like(Wq, 0x7F)
    _, a3 = dg.dg_head_fp8_argmax(x, allnan, scale, choice=c)
    assert a3.tolist() == [-1] * M


def test_head_repeated_calls_reset_ticket(cuda_device):
    x, Wq, scale = S.head_inputs(4, 10000, 1024, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_HEAD_FP8_ARGMAX, 4, 10000, 1024)
    outs = [dg.dg_head_fp8_argmax(x, Wq, scale, ws=ws) for _ in range(5)]
    for l, a in outs[1:]:
        assert torch.equal(l.view(torch.int16), outs[0][0].view(torch.int16)) and torch.equal(a, outs[0][1])
    assert dg.dg_device_status(ws) == 0
