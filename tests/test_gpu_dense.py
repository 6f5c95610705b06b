"""GPU parity of the bf16 linear and the fused gate/up against the fp64 oracle."""
import itertools

import numpy as np
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import oracle as O
from oracle import tolerance as T
from synth import decode_inputs as S
from tests._helpers import bits16, f64, sample_rows, lin_excess, silu_excess

pytestmark = pytest.mark.gpu

SWEEP_NK = [(4096, 4096), (12288, 4096), (4096, 12288), (32768, 1024), (8192, 4096)]
SWEEP_M = [1, 2, 4, 8, 16, 32, 64, 128]
GATE_UP_M = [1, 2, 3, 4, 6, 8, 12, 16, 32, 64, 128]


def _lin_check(x, W, y, rows=None):
    xb = bits16(x)
    Wb = bits16(W if rows is None else W[torch.as_tensor(rows, device=W.device)])
    ref, ad = O.linear_bf16(xb, Wb)
    got = f64(y if rows is None else y[:, torch.as_tensor(rows, device=y.device)])
    exc = lin_excess(got, ref, ad)
    assert (exc <= 0).all(), f"max excess {exc.max():.3e} at {np.unravel_index(exc.argmax(), exc.shape)}"


CC = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0)
BULK = dg.Choice.make(dg.DG_VAR_CC_BULK, 0, 0, 0)
TC = dg.Choice.make(dg.DG_VAR_TC, 0)
MMA = dg.Choice.make(dg.DG_VAR_MMA, 0, 0, 0, 0)
FAMILIES = {"cc": CC, "bulk": BULK, "tc": TC, "mma": MMA, "default": None}
SMALL = [(1, 2048, 1024), (3, 130, 1040), (5, 77, 520), (8, 300, 2056), (16, 96, 264), (37, 65, 136),
         (128, 64, 1024), (2, 1, 8), (16, 1000, 4096), (64, 300, 3000), (100, 257, 1096), (128, 640, 6144)]


@pytest.mark.parametrize("family", ["cc", "bulk", "tc", "default"])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_gemv_small_exhaustive(cuda_device, M, N, K, family):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K)
    y = dg.dg_gemv_bf16(x, W, ws=ws, choice=FAMILIES[family])
    torch.cuda.synchronize()
    _lin_check(x, W, y)
    assert dg.dg_device_status(ws) == 0


@pytest.mark.parametrize("N,K", SWEEP_NK)
@pytest.mark.parametrize("M", SWEEP_M)
def test_gemv_sweep_full_size_sampled(cuda_device, M, N, K):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    y = dg.dg_gemv_bf16(x, W)
    torch.cuda.synchronize()
    _lin_check(x, W, y, rows=sample_rows(N, 96, seed=N + K + M))


def _variants(op, mt_max):
    """Every CUDA-core variant: register-streamed (rows/warp, warps/CTA, CTA cap, warps
    sharing a row group's K segments) and bulk-staged (pipeline depth, CTAs per SM).
    All share one arithmetic."""
    out = []
    for R, wpc, cap in itertools.product((1, 2, 4, 8), (2, 4, 8), (0, 1)):
        if op == dg.DG_OP_GATE_UP_SILU and R < 2:
            continue
        for ks in sorted({1, 2, wpc}):
            out.append(dg.Choice.make(dg.DG_VAR_CC_WARP, R, wpc, cap, ks if ks > 1 else 0))
    for st, cps in itertools.product((0, 2, 3, 8), (1, 2)):
        out.append(dg.Choice.make(dg.DG_VAR_CC_BULK, 0, st, cps))
    return out


@pytest.mark.parametrize("M,N,K", [(1, 1000, 3080), (2, 300, 8200), (1, 77, 520), (3, 515, 1024), (8, 256, 4096),
                                   (13, 70, 2048)])
def test_gemv_cc_variants_bitwise_identical(cuda_device, M, N, K):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ref = dg.dg_gemv_bf16(x, W, choice=CC)
    for c in _variants(dg.DG_OP_GEMV_BF16, 8):
        try:
            y = dg.dg_gemv_bf16(x, W, choice=c)
        except dg.DGError as e:            # a depth that does not fit shared memory for this K
            assert e.status in (3, 8) and c.variant == dg.DG_VAR_CC_BULK, (repr(c), e.status)
            continue
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), repr(c)
    for _ in range(3):
        assert torch.equal(dg.dg_gemv_bf16(x, W, choice=CC).view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(16, 4096, 4096), (40, 1000, 3080), (128, 768, 2048), (6, 32768, 1024)])
def test_gemv_tc_variants_bitwise_identical(cuda_device, M, N, K):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K)
    ref = dg.dg_gemv_bf16(x, W, ws=ws, choice=TC)
    for st in (2, 3, 4, 5, 6):
        c = dg.Choice.make(dg.DG_VAR_TC, st)
        try:
            y = dg.dg_gemv_bf16(x, W, ws=ws, choice=c)
        except dg.DGError as e:            # a depth that does not fit shared memory for this M
            assert e.status == 8
            continue
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), st
    for _ in range(3):
        assert torch.equal(dg.dg_gemv_bf16(x, W, ws=ws, choice=TC).view(torch.int16), ref.view(torch.int16))
    assert dg.dg_device_status(ws) == 0


@pytest.mark.parametrize("family", ["cc", "bulk", "tc"])
def test_gemv_identity_and_one_hot_exact(cuda_device, family):
    c = FAMILIES[family]
    K = 1040
    eye = torch.eye(K, dtype=torch.bfloat16, device=cuda_device)
    for M in (5, 40):
        x, W = S.linear_inputs(M, 300, K, device=cuda_device)
        assert torch.equal(dg.dg_gemv_bf16(x, eye, choice=c).view(torch.int16), x.view(torch.int16))
    for k in (0, 517, K - 1):
        e = torch.zeros((1, K), dtype=torch.bfloat16, device=cuda_device)
        e[0, k] = 1.0
        y = dg.dg_gemv_bf16(e, W, choice=c)
        assert torch.equal(y[0].view(torch.int16), W[:, k].contiguous().view(torch.int16))


def test_gemv_writes_nothing_outside_y(cuda_device):
    M, N, K = 3, 77, 520
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    buf = torch.full((M * N + 64,), 12345, dtype=torch.int16, device=cuda_device)
    y = buf[8:8 + M * N].view(torch.bfloat16).view(M, N)   # 16-byte aligned view
    dg.dg_gemv_bf16(x, W, y=y)
    torch.cuda.synchronize()
    assert (buf[:8] == 12345).all() and (buf[8 + M * N:] == 12345).all()
    _lin_check(x, W, y)


# ---------------------------------------------------------------- gate/up

def _gate_up_check(x, Wgu, out, cols=None):
    Nh = Wgu.shape[0] // 2
    if cols is None:
        r = O.gate_up_silu(bits16(x), bits16(Wgu))
        got = f64(out)
    else:
        c = torch.as_tensor(cols, device=Wgu.device)
        rows = torch.stack((2 * c, 2 * c + 1), dim=1).reshape(-1)
        r = O.gate_up_silu(bits16(x), bits16(Wgu[rows]))
        got = f64(out[:, c])
    exc = silu_excess(got, r["g"], r["u"], r["absg"], r["absu"], r["out"])
    assert (exc <= 0).all(), f"max excess {exc.max():.3e}"


@pytest.mark.parametrize("family", ["cc", "bulk", "tc", "default"])
@pytest.mark.parametrize("M,Nh,K", [(1, 96, 1024), (3, 65, 1040), (6, 200, 520), (12, 33, 2048), (64, 16, 264),
                                    (16, 700, 4096), (128, 96, 1544)])
def test_gate_up_small_exhaustive(cuda_device, M, Nh, K, family):
    x, Wgu = S.gate_up_inputs(M, Nh, K, device=cuda_device)
    out = dg.dg_gate_up_silu(x, Wgu, choice=FAMILIES[family])
    torch.cuda.synchronize()
    _gate_up_check(x, Wgu, out)


@pytest.mark.parametrize("M", GATE_UP_M)
def test_gate_up_full_size_sampled(cuda_device, M):
    x, Wgu = S.gate_up_inputs(M, 12288, 4096, device=cuda_device)
    out = dg.dg_gate_up_silu(x, Wgu)
    torch.cuda.synchronize()
    _gate_up_check(x, Wgu, out, cols=sample_rows(12288, 64, seed=M))


@pytest.mark.parametrize("M,K", [(1, 5128), (2, 3080), (6, 2056)])
def test_gate_up_variants_bitwise_identical(cuda_device, M, K):
    x, Wgu = S.gate_up_inputs(M, 300, K, device=cuda_device)
    ref = dg.dg_gate_up_silu(x, Wgu, choice=CC)
    for c in _variants(dg.DG_OP_GATE_UP_SILU, 8):
        try:
            out = dg.dg_gate_up_silu(x, Wgu, choice=c)
        except dg.DGError as e:
            assert e.status in (3, 8) and c.variant == dg.DG_VAR_CC_BULK, (repr(c), e.status)
            continue
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), repr(c)
    x, Wgu = S.gate_up_inputs(32, 3000, 4096, device=cuda_device)
    ref = dg.dg_gate_up_silu(x, Wgu, choice=TC)
    for st in (2, 3, 4, 5):
        out = dg.dg_gate_up_silu(x, Wgu, choice=dg.Choice.make(dg.DG_VAR_TC, st))
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), st


def test_gate_up_matches_two_linears_plus_silu_on_device(cuda_device):
    """out == bf16(silu(g)*u) with g, u the exact fp32 dot products: one-hot rows make g, u exact."""
    K, Nh = 64, 8
    Wf = torch.zeros((2 * Nh, K))
    for j in range(Nh):
        Wf[2 * j, j] = 1.0
        Wf[2 * j + 1, 32 + j] = 1.0
    x = torch.randn((2, K), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    g = x.float()[:, :Nh]
    u = x.float()[:, 32:32 + Nh]
    ref = (g / (1 + torch.exp(-g)) * u)
    for c in (CC, BULK, TC):
        out = dg.dg_gate_up_silu(x.to(cuda_device), Wf.to(torch.bfloat16).to(cuda_device), choice=c)
        assert torch.allclose(out.float().cpu(), ref, rtol=2 ** -7, atol=1e-6)


# ---------------------------------------------------------------- argument errors on device

def test_bad_arguments_are_rejected_before_launch(cuda_device):
    x, W = S.linear_inputs(2, 64, 256, device=cuda_device)
    y = torch.empty((2, 64), dtype=torch.bfloat16, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, 2, 64, 256)
    x2, W2 = S.linear_inputs(2, 64, 250, device=cuda_device)       # K not a multiple of 8
    with pytest.raises(dg.DGError) as e:
        dg.dg_gemv_bf16(x2, W2, y, ws=ws)
    assert e.value.status == 3
    raw = torch.empty(2 * 64 + 1, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(dg.DGError) as e:                           # output not 16-byte aligned
        dg.dg_gemv_bf16(x, W, raw[1:].view(2, 64), ws=ws)
    assert e.value.status == 2
    with pytest.raises(dg.DGError) as e:                           # workspace too small
        dg.dg_gemv_bf16(x, W, y, ws=ws[:8])
    assert e.value.status == 4
    torch.cuda.synchronize()


def test_launch_without_pdl_gives_same_bits(cuda_device):
    """Programmatic dependent launch changes scheduling only, never results."""
    cases = [(dg.dg_gemv_bf16, S.linear_inputs(3, 1000, 2048, device=cuda_device), CC),
             (dg.dg_gemv_bf16, S.linear_inputs(40, 1000, 2048, device=cuda_device), TC),
             (dg.dg_gate_up_silu, S.gate_up_inputs(20, 300, 1024, device=cuda_device), TC)]
    assert dg.dg_launch_flags() == dg.DG_LAUNCH_PDL
    ref = [f(x, W, choice=c) for f, (x, W), c in cases]
    dg.dg_set_launch_flags(0)
    try:
        got = [f(x, W, choice=c) for f, (x, W), c in cases]
    finally:
        dg.dg_set_launch_flags(dg.DG_LAUNCH_PDL)
    for r, g in zip(ref, got):
        assert torch.equal(r.view(torch.int16), g.view(torch.int16))
    # back-to-back dependent calls: the second reads the first's output
    x, W = S.linear_inputs(4, 1024, 1024, device=cuda_device)
    y1 = dg.dg_gemv_bf16(x, W, choice=CC)
    y2 = dg.dg_gemv_bf16(y1, W, choice=CC)
    torch.cuda.synchronize()
    _lin_check(y1, W, y2)


# ------------------------------------------------------------------ mid-M (129..512)

MID_M = [129, 200, 256, 300, 512]


@pytest.mark.parametrize("family", ["tc", "default"])
@pytest.mark.parametrize("M,N,K", [(129, 300, 1040), (200, 640, 2056), (256, 257, 1096), (300, 130, 520),
                                   (512, 384, 3080)])
def test_gemv_mid_m_small(cuda_device, M, N, K, family):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K)
    y = dg.dg_gemv_bf16(x, W, ws=ws, choice=FAMILIES[family])
    torch.cuda.synchronize()
    _lin_check(x, W, y)
    assert dg.dg_device_status(ws) == 0


@pytest.mark.parametrize("N,K", [(32768, 1024), (8192, 1024), (4096, 12288)])
@pytest.mark.parametrize("M", [192, 256, 512])
def test_gemv_mid_m_full_size_sampled(cuda_device, M, N, K):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    y = dg.dg_gemv_bf16(x, W)
    torch.cuda.synchronize()
    _lin_check(x, W, y, rows=sample_rows(N, 48, seed=N + K + M))


@pytest.mark.parametrize("M,N,K", [(200, 1000, 3080), (256, 4096, 4096)])
def test_gemv_mid_m_tc_variants_bitwise_identical(cuda_device, M, N, K):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ref = dg.dg_gemv_bf16(x, W, choice=TC)
    for st in (2, 3, 4, 5, 8):
        try:
            y = dg.dg_gemv_bf16(x, W, choice=dg.Choice.make(dg.DG_VAR_TC, st))
        except dg.DGError as e:            # a depth whose ring cannot hold the 256-token tile
            assert e.status == 8, (st, e.status)
            continue
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), st
    # the CUDA-core family computes the same outputs within the tolerance
    yc = dg.dg_gemv_bf16(x, W, choice=CC)
    torch.cuda.synchronize()
    _lin_check(x, W, yc, rows=sample_rows(N, 32, seed=M))


# 256-token tiles on more tiles than SMs run two tiles per CTA (one wave); 153 tiles
# gives an odd last CTA, +40 rows a partial last tile.
# Tile counts at which the tensor-core K-split takes each cluster width from 1 to 8 ranks,
# including the counts where one wave of clusters caps it below SMs x CTAs per SM / tiles
# (37-38, 39-43, 47-50, 59-60, 75-76, 98-101 tiles at two CTAs per SM; 16 and 24 tiles at
# one), the last tile ragged.
SPLIT_TILES = [1, 3, 5, 7, 16, 24, 38, 43, 48, 60, 76, 100]


@pytest.mark.parametrize("K", [1024, 4096 + 64])
@pytest.mark.parametrize("tiles", SPLIT_TILES)
@pytest.mark.parametrize("M", [16, 100, 200])
def test_gemv_tc_every_split_width(cuda_device, M, tiles, K):
    """The tensor-core linear at every K-split width the rule picks (one per tile count
    above), against the oracle on sampled rows, and bit for bit across ring depths."""
    N = 128 * tiles - 24
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K)
    y = dg.dg_gemv_bf16(x, W, ws=ws, choice=TC)
    torch.cuda.synchronize()
    assert dg.dg_device_status(ws) == 0
    _lin_check(x, W, y, rows=sample_rows(N, 24, seed=N + K + M))
    y3 = dg.dg_gemv_bf16(x, W, choice=dg.Choice.make(dg.DG_VAR_TC, 3))
    assert torch.equal(y3.view(torch.int16), y.view(torch.int16))


PAIR_N = [128 * 153, 128 * 153 + 40]


@pytest.mark.parametrize("K", [64, 1040])
@pytest.mark.parametrize("N", PAIR_N)
@pytest.mark.parametrize("M", [129, 256, 300])
def test_gemv_mid_m_paired_tiles(cuda_device, M, N, K):
    """Paired tiles against the oracle (rows of the odd last CTA included), against one
    tile per CTA bit for bit (the first 152 tiles alone take that path with the same
    unsplit chain, for the first 256 token rows), and across pipeline depths."""
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    y = dg.dg_gemv_bf16(x, W)
    rows = np.unique(np.concatenate([sample_rows(N, 40, seed=N + K + M), np.arange(N - 130, N)]))
    torch.cuda.synchronize()
    _lin_check(x, W, y, rows=rows)
    n1 = 128 * 152
    y1 = dg.dg_gemv_bf16(x, W[:n1].contiguous())
    m1 = min(M, 256)          # (rows past 256 are a second chunk of fewer tokens, with its own split rule)
    assert torch.equal(y[:m1, :n1].contiguous().view(torch.int16), y1[:m1].contiguous().view(torch.int16))
    for st in (2, 3):
        y2 = dg.dg_gemv_bf16(x, W, choice=dg.Choice.make(dg.DG_VAR_TC, st))
        assert torch.equal(y2.view(torch.int16), y.view(torch.int16)), st


def test_gemv_mid_m_paired_tiles_one_hot_exact(cuda_device):
    """x = e_k rows: every output of both tiles of every CTA equals W[n, k] exactly."""
    N, K, M = 128 * 153 + 40, 1040, 256
    _, W = S.linear_inputs(1, N, K, device=cuda_device)
    ks = [(37 * m + 5) % K for m in range(M)]
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=cuda_device)
    for m, k in enumerate(ks):
        x[m, k] = 1.0
    y = dg.dg_gemv_bf16(x, W)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), W[:, ks].t().contiguous().view(torch.int16))


@pytest.mark.parametrize("M", [129, 256])
def test_gate_up_mid_m_paired_tiles(cuda_device, M):
    Nh = 64 * 153 + 20                 # 2 * Nh = 19624 rows: 154 tiles
    x, Wgu = S.gate_up_inputs(M, Nh, 1040, device=cuda_device)
    out = dg.dg_gate_up_silu(x, Wgu)
    torch.cuda.synchronize()
    cols = np.unique(np.concatenate([sample_rows(Nh, 40, seed=M), np.arange(Nh - 70, Nh)]))
    _gate_up_check(x, Wgu, out, cols=cols)


@pytest.mark.parametrize("M", [160, 384])
def test_gate_up_mid_m(cuda_device, M):
    x, Wgu = S.gate_up_inputs(M, 700, 2056, device=cuda_device)
    out = dg.dg_gate_up_silu(x, Wgu)
    torch.cuda.synchronize()
    _gate_up_check(x, Wgu, out)


# ---------------------------------------------------------------- warp-level tensor cores (mma.sync)

MMA_SMALL = [(3, 130, 1040), (5, 77, 520), (8, 300, 2056), (16, 96, 264), (1, 2048, 1024), (2, 1, 8),
             (12, 1000, 4096), (9, 257, 1096), (16, 640, 6144), (4, 33, 4104), (15, 4099, 520)]


@pytest.mark.parametrize("M,N,K", MMA_SMALL)
def test_gemv_mma_small_exhaustive(cuda_device, M, N, K):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    y = dg.dg_gemv_bf16(x, W, choice=MMA)
    torch.cuda.synchronize()
    _lin_check(x, W, y)


@pytest.mark.parametrize("N,K", SWEEP_NK)
@pytest.mark.parametrize("M", [3, 4, 8, 12, 16])
def test_gemv_mma_full_size_sampled(cuda_device, M, N, K):
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    y = dg.dg_gemv_bf16(x, W, choice=MMA)
    torch.cuda.synchronize()
    _lin_check(x, W, y, rows=sample_rows(N, 96, seed=N + K + 7 * M))


@pytest.mark.parametrize("M,N,K", [(3, 1000, 3080), (8, 300, 8200), (12, 77, 520), (16, 515, 1024), (5, 4096, 4096),
                                   (9, 70, 2048)])
def test_gemv_mma_variants_bitwise_identical(cuda_device, M, N, K):
    """Every geometry of the warp-level tensor-core family (warps sharing a group's
    segments, warps per CTA, CTA cap, chunks per load round) gives the same bits."""
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ref = dg.dg_gemv_bf16(x, W, choice=MMA)
    for ks, wpc, cap, u in itertools.product((1, 2, 4, 8), (4, 8), (0, 1), (2, 4, 8)):
        if ks > wpc:
            continue
        y = dg.dg_gemv_bf16(x, W, choice=dg.Choice.make(dg.DG_VAR_MMA, ks, wpc, cap, u))
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (ks, wpc, cap, u)
    for _ in range(3):
        assert torch.equal(dg.dg_gemv_bf16(x, W, choice=MMA).view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("M,Nh,K", [(3, 96, 1040), (8, 300, 4096), (12, 12288, 4096), (16, 77, 2064)])
def test_gate_up_mma(cuda_device, M, Nh, K):
    x, Wgu = S.gate_up_inputs(M, Nh, K, device=cuda_device)
    out = dg.dg_gate_up_silu(x, Wgu, choice=MMA)
    torch.cuda.synchronize()
    _gate_up_check(x, Wgu, out, cols=None if Nh <= 1000 else sample_rows(Nh, 96, seed=M))
    for ks, wpc, u in ((1, 8, 4), (8, 8, 2), (2, 4, 8)):
        o2 = dg.dg_gate_up_silu(x, Wgu, choice=dg.Choice.make(dg.DG_VAR_MMA, ks, wpc, 0, u))
        assert torch.equal(o2.view(torch.int16), out.view(torch.int16)), (ks, wpc, u)


def test_mma_refuses_more_than_16_rows(cuda_device):
    x, W = S.linear_inputs(17, 64, 64, device=cuda_device)
    with pytest.raises(dg.DGError) as e:
        dg.dg_gemv_bf16(x, W, choice=MMA)
    assert e.value.status == 3
