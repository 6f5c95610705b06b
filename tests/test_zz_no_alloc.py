"""The head entry point for callers that cannot allocate device memory.

dg_head_fp8_argmax_noalloc keeps its scratch in a static device array inside the
library, for engines and plugins that are not allowed to call cudaMalloc.  This file
is collected last so that a run stopping at its first failure has already run every
other test; it passes alone in a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import tolerance as T
from oracle import oracle as O
from synth import decode_inputs as S
from tests._helpers import bits16, f64, sample_rows, lin_excess, silu_excess

pytestmark = pytest.mark.gpu

# every kernel family and geometry the head's selection may run
CHOICES = {
    "default": None,
    "cc_warp": dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0),
    "cc_bulk": dg.Choice.make(dg.DG_VAR_CC_BULK, 0, 0, 0),
    "cc_bulk_2cta": dg.Choice.make(dg.DG_VAR_CC_BULK, 0, 0, 2),
    "tc": dg.Choice.make(dg.DG_VAR_TC, 0),
}


def _noalloc(x, Wq, scale, logits, argmax, choice=None):
    """Call the C entry point directly through the library's C ABI."""
    P = ctypes.c_void_p
    M, K = x.shape
    N = Wq.shape[0]
    stream = P(torch.cuda.current_stream().cuda_stream)
    return dg.lib().dg_head_fp8_argmax_noalloc(P(x.data_ptr()), P(Wq.data_ptr()), P(scale.data_ptr()),
                                               P(logits.data_ptr()), P(argmax.data_ptr()), M, N, K,
                                               stream, None if choice is None else ctypes.byref(choice))


def _status():
    v = ctypes.c_int32(-1)
    assert dg.lib().dg_head_fp8_argmax_noalloc_status(ctypes.byref(v), None) == 0
    return v.value


def _check_argmax(x, Wq, scale, am):
    """The oracle's own pick on these inputs, unless its top-2 gap is within twice the
    error bound (then any index whose exact logit lies in that window is accepted)."""
    sc = float(scale.cpu()[0])
    xb, Wn = bits16(x), Wq.cpu().numpy()
    idx, _, gap = O.head_argmax(xb, Wn, sc)
    got = am.cpu().numpy()
    for m in range(x.shape[0]):
        if got[m] == idx[m]:
            continue
        lg, ad = O.head_fp8(xb[m:m + 1], Wn, sc, rows=np.array([idx[m], got[m]]))
        window = 2 * (T.REL * ad[0].max() + T.ABS)
        assert gap[m] <= window and lg[0, 0] - lg[0, 1] <= window, (m, got[m], idx[m], gap[m])


@pytest.mark.parametrize("name", list(CHOICES))
@pytest.mark.parametrize("M,N,K", [(1, 248320, 4096), (3, 4099, 1040), (8, 50000, 4096)])
def test_noalloc_head_matches_workspace_entry_point_twice(cuda_device, M, N, K, name):
    choice = CHOICES[name]
    x, Wq, scale = S.head_inputs(M, N, K, device=cuda_device)
    ref_logits, ref_am = dg.dg_head_fp8_argmax(x, Wq, scale, choice=choice)
    for _ in range(2):                       # two calls in a row share the static scratch
        logits = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda_device)
        am = torch.full((M,), -7, dtype=torch.int32, device=cuda_device)
        assert _noalloc(x, Wq, scale, logits, am, choice) == 0
        torch.cuda.synchronize()
        assert _status() == 0
        # within the head tests' bound of the oracle's logits (sampled rows)
        rows = sample_rows(N, 64, seed=M)
        sel = torch.as_tensor(rows, device=cuda_device)
        lg, ad = O.head_fp8(bits16(x), Wq[sel].cpu().numpy(), float(scale.cpu()[0]))
        exc = lin_excess(f64(logits[:, sel]), lg, ad)
        assert (exc <= 0).all()
        # the same kernel runs, so every logit and pick has the workspace entry point's bits
        assert torch.equal(logits.view(torch.int16), ref_logits.view(torch.int16))
        assert torch.equal(am, ref_am)
    if M == 1 and name == "default":
        _check_argmax(x, Wq, scale, am)


def test_noalloc_status_reports_a_wait_that_gave_up(cuda_device):
    """The status word of the static scratch is readable: a bounded wait run on the
    scratch that gives up shows as DG_DEVERR_WAIT_TIMEOUT, a refused call leaves it
    alone (it queues nothing, not even its clearing memset), and the next accepted
    call starts from zero again."""
    addr = ctypes.c_void_p(0)
    assert dg.lib().dg_head_fp8_argmax_noalloc_scratch(ctypes.byref(addr)) == 0 and addr.value
    assert dg.lib().dg_selftest_wait_timeout(addr, 2000, None) == 0
    torch.cuda.synchronize()
    assert _status() & dg.DG_DEVERR_WAIT_TIMEOUT
    x, Wq, scale = S.head_inputs(2, 4099, 1040, device=cuda_device)
    logits = torch.empty((2, 4099), dtype=torch.bfloat16, device=cuda_device)
    am = torch.empty((2,), dtype=torch.int32, device=cuda_device)
    bad = dg.Choice.make(dg.DG_VAR_TC, 99)          # refused after the argument checks
    assert _noalloc(x, Wq, scale, logits, am, bad) == dg.DG_ERR_BAD_VARIANT
    torch.cuda.synchronize()
    assert _status() & dg.DG_DEVERR_WAIT_TIMEOUT
    assert _noalloc(x, Wq, scale, logits, am) == 0
    torch.cuda.synchronize()
    assert _status() == 0
    ref_logits, ref_am = dg.dg_head_fp8_argmax(x, Wq, scale)
    assert torch.equal(logits.view(torch.int16), ref_logits.view(torch.int16)) and torch.equal(am, ref_am)


def test_noalloc_rejects_bad_arguments_without_launching(cuda_device):
    x, Wq, scale = S.head_inputs(2, 128, 64, device=cuda_device)
    logits = torch.empty((2, 128), dtype=torch.bfloat16, device=cuda_device)
    am = torch.empty((2,), dtype=torch.int32, device=cuda_device)
    x9 = torch.zeros((9, 64), dtype=torch.bfloat16, device=cuda_device)
    assert _noalloc(x9, Wq, scale, torch.empty((9, 128), dtype=torch.bfloat16, device=cuda_device),
                    torch.empty((9,), dtype=torch.int32, device=cuda_device)) == 1
    raw = torch.empty(2 * 128 + 1, dtype=torch.bfloat16, device=cuda_device)
    assert _noalloc(x, Wq, scale, raw[1:].view(2, 128), am) == 2
    assert _noalloc(x, Wq, scale, logits, am) == 0
    torch.cuda.synchronize()
