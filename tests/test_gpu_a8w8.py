"""GPU parity of the A8W8 block-scaled linear with the fused activation quantisation.

The quantisation decides integers (the e4m3 codes) in binary32 on both sides, so the
codes and the per-(token, block) scales must equal the oracle's bit for bit; the
product is held to the linear error bound against the oracle's fp64 sum over the
same codes.
"""
import numpy as np
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import oracle as O
from oracle import tolerance as T
from synth import decode_inputs as S
from tests._helpers import bits16, f64, sample_rows, lin_excess, silu_excess

pytestmark = pytest.mark.gpu

A8_NK = [(32768, 1024), (8192, 4096)]
A8_M = [1, 2, 4, 8, 16, 32, 64]
SMALL = [(1, 2048, 1024), (3, 130, 1040), (5, 77, 528), (8, 300, 2064), (16, 96, 272), (17, 65, 144),
         (33, 640, 4096), (2, 1, 16), (64, 257, 1040), (64, 128, 8192), (12, 1000, 12288)]


def _wide_x(M, K, seed, device):
    """bf16 activations whose 128-blocks span many magnitudes, with an all-zero block,
    a lone spike and a subnormal-range block."""
    g = torch.Generator().manual_seed(seed)
    nb = (K + 127) // 128
    x = torch.randn((M, K), generator=g)
    x *= torch.exp2(torch.randint(-30, 14, (M, nb), generator=g).float()).repeat_interleave(128, 1)[:, :K]
    if K >= 256:
        x[0, 128:256] = 0.0
        x[-1, 130] = 6.0e4
    if K >= 384:
        x[M // 2, 256:384] *= 2.0 ** -120
    return x.to(torch.bfloat16).to(device)


def _check(x, Wq, sw, y, rows=None):
    r = O.a8w8_linear(bits16(x), Wq.cpu().numpy(), sw.cpu().numpy(), rows=rows)
    got = f64(y if rows is None else y[:, torch.as_tensor(rows, device=y.device)])
    exc = lin_excess(got, r["y"], r["absdot"])
    assert (exc <= 0).all(), f"max excess {exc.max():.3e} at {np.unravel_index(exc.argmax(), exc.shape)}"


@pytest.mark.parametrize("M,K,seed", [(1, 1024, 1), (5, 1040, 2), (64, 4096, 3), (3, 16, 4), (200, 272, 5)])
def test_quant_codes_and_scales_bit_exact(cuda_device, M, K, seed):
    x = _wide_x(M, K, seed, cuda_device)
    q, sx = dg.dg_quant_a8_blockscale(x)
    torch.cuda.synchronize()
    q_ref, sx_ref = O.a8_quant(bits16(x))
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))


@pytest.mark.parametrize("pq", [0, 1])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_a8w8_small_exhaustive(cuda_device, M, N, K, pq):
    _, Wq, sw = S.a8w8_inputs(1, N, K, device=cuda_device)
    x = _wide_x(M, K, M + N + K, cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_A8W8, M, N, K)
    y = dg.dg_gemv_a8w8_blockscale(x, Wq, sw, ws=ws, choice=dg.Choice.make(dg.DG_VAR_TC, 0, pq))
    torch.cuda.synchronize()
    _check(x, Wq, sw, y)
    assert dg.dg_device_status(ws) == 0


@pytest.mark.parametrize("N,K", A8_NK)
@pytest.mark.parametrize("M", A8_M)
def test_a8w8_full_size_sampled(cuda_device, M, N, K):
    x, Wq, sw = S.a8w8_inputs(M, N, K, device=cuda_device)
    y = dg.dg_gemv_a8w8_blockscale(x, Wq, sw)
    torch.cuda.synchronize()
    _check(x, Wq, sw, y, rows=sample_rows(N, 96, seed=N + K + M))


@pytest.mark.parametrize("M,N,K", [(1, 8192, 4096), (16, 32768, 1024), (40, 700, 2064), (64, 8192, 4096),
                                   (3, 130, 1040)])
def test_a8w8_variants_bitwise_identical(cuda_device, M, N, K):
    """Pipeline depth, and the quantisation fused or run as a launch of its own (codes
    streamed by TMA), give the same bits."""
    x, Wq, sw = S.a8w8_inputs(M, N, K, device=cuda_device)
    ref = dg.dg_gemv_a8w8_blockscale(x, Wq, sw)
    for pq in (0, 1):
        for st in [0] + list(range(2, 9)):
            try:
                y = dg.dg_gemv_a8w8_blockscale(x, Wq, sw, choice=dg.Choice.make(dg.DG_VAR_TC, st, pq))
            except dg.DGError as e:
                assert e.status in (3, 8), (st, pq, e.status)
                continue
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (st, pq)


@pytest.mark.parametrize("tiles", [7, 38, 42, 48, 60, 100])
@pytest.mark.parametrize("M", [16, 64])
def test_a8w8_every_split_width(cuda_device, M, tiles):
    """The A8W8 K-split at the tile counts where one wave of clusters sets its width,
    against the oracle on sampled rows."""
    N, K = 128 * tiles - 40, 4096
    x, Wq, sw = S.a8w8_inputs(M, N, K, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_A8W8, M, N, K)
    y = dg.dg_gemv_a8w8_blockscale(x, Wq, sw, ws=ws)
    torch.cuda.synchronize()
    assert dg.dg_device_status(ws) == 0
    _check(x, Wq, sw, y, rows=sample_rows(N, 24, seed=N + M))


@pytest.mark.parametrize("N,K", [(8192, 4096), (300, 1040)])
def test_a8w8_rows_independent_of_the_batch(cuda_device, N, K):
    """The K-split is fixed by (N, K), so a row's bits do not depend on M or on the
    other rows (any prefix, and a permutation)."""
    x, Wq, sw = S.a8w8_inputs(64, N, K, device=cuda_device)
    full = dg.dg_gemv_a8w8_blockscale(x, Wq, sw)
    for M in range(1, 64):
        y = dg.dg_gemv_a8w8_blockscale(x[:M].contiguous(), Wq, sw)
        assert torch.equal(y.view(torch.int16), full[:M].view(torch.int16)), M
    p = torch.randperm(64, generator=torch.Generator().manual_seed(N)).to(cuda_device)
    y = dg.dg_gemv_a8w8_blockscale(x[p].contiguous(), Wq, sw)
    assert torch.equal(y.view(torch.int16), full[p].view(torch.int16))


def test_a8w8_one_hot_and_zero_rows(cuda_device):
    """x = v e_k quantises to a single +-448 code: y[n] = sx * sw * 448 * w[n, k];
    an all-zero row gives zeros."""
    N, K = 260, 384
    _, Wq, sw = S.a8w8_inputs(1, N, K, device=cuda_device)
    x = torch.zeros((3, K), dtype=torch.bfloat16, device=cuda_device)
    x[0, 5] = 3.25
    x[1, 383] = -1500.0
    y = dg.dg_gemv_a8w8_blockscale(x, Wq, sw)
    torch.cuda.synchronize()
    _check(x, Wq, sw, y)
    assert (y[2] == 0).all()


def test_a8w8_graph_replay_and_no_sync(cuda_device):
    M, N, K = 8, 8192, 4096
    x, Wq, sw = S.a8w8_inputs(M, N, K, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_A8W8, M, N, K)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=cuda_device)
    ref = dg.dg_gemv_a8w8_blockscale(x, Wq, sw).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        dg.dg_gemv_a8w8_blockscale(x, Wq, sw, y=y, ws=ws, stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                dg.dg_gemv_a8w8_blockscale(x, Wq, sw, y=y, ws=ws, stream=s)
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert dg.dg_device_status(ws) == 0


def test_a8w8_argument_errors_launch_nothing(cuda_device):
    x, Wq, sw = S.a8w8_inputs(2, 300, 1040, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_A8W8, 2, 300, 1040)
    with pytest.raises(dg.DGError) as e:                     # workspace too small
        dg.dg_gemv_a8w8_blockscale(x, Wq, sw, ws=ws[:1024])
    assert e.value.status == dg.DG_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(dg.DGError) as e:                     # a CUDA-core variant does not exist here
        dg.dg_gemv_a8w8_blockscale(x, Wq, sw, choice=dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8))
    assert e.value.status == dg.DG_ERR_BAD_VARIANT
    K = 32768                                                # more K-blocks per rank than the kernel holds
    xl, Wl, swl = S.a8w8_inputs(1, 128, K, device=cuda_device)
    with pytest.raises(dg.DGError) as e:
        dg.dg_gemv_a8w8_blockscale(xl, Wl, swl)
    assert e.value.status == dg.DG_ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert dg.dg_device_status(ws) == 0
