"""Failure reporting on the device without a fault: a bounded wait that runs out
sets the status word and returns, after which the context still computes; host
argument checks refuse bad calls before any launch."""
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import oracle as O
from oracle import tolerance as T
from synth import decode_inputs as S
from tests._helpers import bits16, f64, lin_excess, silu_excess

pytestmark = pytest.mark.gpu


def test_wait_timeout_sets_status_and_context_survives(cuda_device):
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, 1, 64, 64)
    assert dg.dg_device_status(ws) == 0
    dg.dg_selftest_wait_timeout(ws, timeout_us=20000)
    torch.cuda.synchronize()
    assert dg.dg_device_status(ws) & dg.DG_DEVERR_WAIT_TIMEOUT
    dg.dg_device_status_clear(ws)
    assert dg.dg_device_status(ws) == 0
    # the same workspace and the same context keep computing correctly
    x, W = S.linear_inputs(4, 640, 2048, device=cuda_device)
    for choice in (None, dg.Choice.make(dg.DG_VAR_TC, 0)):
        y = dg.dg_gemv_bf16(x, W, ws=dg.workspace(dg.DG_OP_GEMV_BF16, 4, 640, 2048), choice=choice)
        torch.cuda.synchronize()
        ref, ad = O.linear_bf16(bits16(x), bits16(W))
        assert (lin_excess(f64(y), ref, ad) <= 0).all()


def test_wait_timeout_argument_checks(cuda_device):
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, 1, 64, 64)
    for bad in (0, -5, 2000001):
        with pytest.raises(dg.DGError) as e:
            dg.dg_selftest_wait_timeout(ws, timeout_us=bad)
        assert e.value.status == dg.DG_ERR_INVALID_ARG
    with pytest.raises(dg.DGError) as e:
        dg.dg_selftest_wait_timeout(ws[4:], timeout_us=100)
    assert e.value.status == dg.DG_ERR_ALIGNMENT


def test_bad_calls_refused_before_launch(cuda_device):
    x, W = S.linear_inputs(2, 64, 64, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_GEMV_BF16, 2, 64, 64)
    with pytest.raises(dg.DGError) as e:           # workspace too small
        dg.dg_gemv_bf16(x, W, ws=ws[:64])
    assert e.value.status == dg.DG_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(dg.DGError) as e:           # K not a multiple of 8
        xb = torch.zeros((2, 60), dtype=torch.bfloat16, device=cuda_device)
        Wb = torch.zeros((64, 60), dtype=torch.bfloat16, device=cuda_device)
        dg.dg_gemv_bf16(xb, Wb, ws=ws)
    assert e.value.status in (dg.DG_ERR_ALIGNMENT, dg.DG_ERR_UNSUPPORTED_SHAPE)
    with pytest.raises(dg.DGError) as e:           # unknown variant
        dg.dg_gemv_bf16(x, W, ws=ws, choice=dg.Choice.make(9, 0))
    assert e.value.status == dg.DG_ERR_BAD_VARIANT
    torch.cuda.synchronize()
    assert dg.dg_device_status(ws) == 0
