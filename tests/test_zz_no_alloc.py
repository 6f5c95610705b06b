"""The head entry point for callers that cannot allocate device memory.

dg_head_fp8_argmax_noalloc keeps its scratch in a static device array inside the
library, for engines and plugins that are not allowed to call cudaMalloc.  This file
is collected last so that a run stopping at its first failure has already run every
other test; it passes alone in a fresh process and after the rest of the suite.
"""
import ctypes

import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import tolerance as T
from oracle import oracle as O
from synth import decode_inputs as S
from tests._helpers import bits16, f64, sample_rows

pytestmark = pytest.mark.gpu


def _noalloc(x, Wq, scale, logits, argmax):
    """Call the C entry point directly through the library's C ABI."""
    P = ctypes.c_void_p
    M, K = x.shape
    N = Wq.shape[0]
    stream = P(torch.cuda.current_stream().cuda_stream)
    return dg.lib().dg_head_fp8_argmax_noalloc(P(x.data_ptr()), P(Wq.data_ptr()), P(scale.data_ptr()),
                                               P(logits.data_ptr()), P(argmax.data_ptr()), M, N, K,
                                               stream, None)


@pytest.mark.parametrize("M,N,K", [(1, 248320, 4096), (3, 4099, 1040), (8, 50000, 4096)])
def test_noalloc_head_matches_workspace_entry_point_twice(cuda_device, M, N, K):
    x, Wq, scale = S.head_inputs(M, N, K, device=cuda_device)
    ref_logits, ref_am = dg.dg_head_fp8_argmax(x, Wq, scale)
    for _ in range(2):                       # two calls in a row share the static scratch
        logits = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=cuda_device)
        am = torch.full((M,), -7, dtype=torch.int32, device=cuda_device)
        assert _noalloc(x, Wq, scale, logits, am) == 0
        torch.cuda.synchronize()
        # within the head tests' bound of the workspace entry point's logits (sampled rows)
        rows = sample_rows(N, 64, seed=M)
        sel = torch.as_tensor(rows, device=cuda_device)
        _, ad = O.head_fp8(bits16(x), Wq[sel].cpu().numpy(), float(scale.cpu()[0]))
        exc = T.linear_excess(f64(logits[:, sel]), f64(ref_logits[:, sel]), ad)
        assert (exc <= 0).all()
        # the same kernel runs, so in fact every logit has the same bits
        assert torch.equal(logits.view(torch.int16), ref_logits.view(torch.int16))
        assert torch.equal(am, ref_am)


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
