"""GPU parity of the small-M MoE W1 (+SiLU.mul) and W2 (+combine), N-split."""
import numpy as np
import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from oracle import oracle as O
from oracle import tolerance as T
from synth import decode_inputs as S
from tests._helpers import bits16, f64, lin_excess, silu_excess

pytestmark = pytest.mark.gpu

E, I, K, TOPK = 128, 1536, 4096, 6
MOE_M = [1, 2, 4, 8, 16]
CC = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0, 0, 2)
TC = dg.Choice.make(dg.DG_VAR_TC, 0)
# the CUDA-core kernels in row-range order (one contiguous row range of every expert per CTA)
RANGE = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0, 0, 0, 2)
FAMILIES = {"cc": CC, "tc": TC, "range": RANGE, "default": None}
RANGE_W2_MAX_M = 10        # every pair's activation row of the call fits in shared memory


@pytest.fixture(scope="module")
def moe_w(cuda_device):
    return S.moe_weights(E, I, K, K, device=cuda_device)


def _compact(ids, *per_expert):
    """Restrict weights to the experts the routing uses (ids renumbered, order kept)."""
    ids_np = ids.cpu().numpy()
    used = np.unique(ids_np[(ids_np >= 0) & (ids_np < E)])
    remap = {int(e): i for i, e in enumerate(used)}
    ids_c = np.vectorize(lambda e: remap.get(int(e), 10 ** 6))(ids_np).astype(np.int32)
    sel = torch.as_tensor(used, device=per_expert[0].device)
    return ids_c, [t[sel].cpu().numpy() for t in per_expert]


def _w1_ref(x, ids, W1q, s1):
    ids_c, (w1, sc1) = _compact(ids, W1q, s1)
    return O.moe_w1_silu(bits16(x), ids_c, w1, sc1)


def _w2_ref(a, ids, gw, W2q, s2):
    ids_c, (w2, sc2) = _compact(ids, W2q, s2)
    return O.moe_w2(bits16(a), ids_c, gw.cpu().numpy(), w2, sc2)


@pytest.mark.parametrize("family", ["cc", "tc", "range"])
@pytest.mark.parametrize("M", MOE_M)
def test_moe_w1_full_size(cuda_device, moe_w, M, family):
    W1q, s1, W2q, s2 = moe_w
    x, ids, gw = S.moe_inputs(M, K, TOPK, E, device=cuda_device)
    ws = dg.workspace(dg.DG_OP_MOE_W1, M, I, K, TOPK)
    a = dg.dg_moe_w1_silu(x, ids, W1q, s1, ws=ws, choice=FAMILIES[family])
    torch.cuda.synchronize()
    r = _w1_ref(x, ids, W1q, s1)
    exc = silu_excess(f64(a), r["g"], r["u"], r["absg"], r["absu"], r["a"])
    assert (exc <= 0).all(), f"max excess {exc.max():.3e}"
    assert dg.dg_device_status(ws) == 0


@pytest.mark.parametrize("family", ["cc", "tc", "range"])
@pytest.mark.parametrize("M", MOE_M)
def test_moe_w2_full_size_on_gpu_activations(cuda_device, moe_w, M, family):
    if family == "range" and M > RANGE_W2_MAX_M:
        pytest.skip("the row-range W2 keeps every pair's row in shared memory")
    W1q, s1, W2q, s2 = moe_w
    c = FAMILIES[family]
    x, ids, gw = S.moe_inputs(M, K, TOPK, E, device=cuda_device)
    a = dg.dg_moe_w1_silu(x, ids, W1q, s1)
    ws = dg.workspace(dg.DG_OP_MOE_W2, M, K, I, TOPK)
    y = dg.dg_moe_w2(a, ids, gw, W2q, s2, ws=ws, choice=c)
    torch.cuda.synchronize()
    ref, bound = _w2_ref(a, ids, gw, W2q, s2)
    exc = lin_excess(f64(y), ref, bound)
    assert (exc <= 0).all(), f"max excess {exc.max():.3e}"
    # repeated calls reuse the workspace tickets and give the same bits
    for _ in range(3):
        assert torch.equal(dg.dg_moe_w2(a, ids, gw, W2q, s2, ws=ws, choice=c).view(torch.int16), y.view(torch.int16))
    assert dg.dg_device_status(ws) == 0


@pytest.mark.parametrize("M", [1, 5, 16])
def test_moe_tc_stages_bitwise_identical(cuda_device, moe_w, M):
    W1q, s1, W2q, s2 = moe_w
    x, ids, gw = S.moe_inputs(M, K, TOPK, E, rep=3, device=cuda_device)
    a_ref = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=TC)
    y_ref = dg.dg_moe_w2(a_ref, ids, gw, W2q, s2, choice=TC)
    for st in (2, 3, 5, 8):
        c = dg.Choice.make(dg.DG_VAR_TC, st)
        assert torch.equal(dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=c).view(torch.int16), a_ref.view(torch.int16))
        assert torch.equal(dg.dg_moe_w2(a_ref, ids, gw, W2q, s2, choice=c).view(torch.int16), y_ref.view(torch.int16))


@pytest.mark.parametrize("M", [1, 4, 16])
def test_moe_tiles_and_warps_bitwise_identical(cuda_device, moe_w, M):
    W1q, s1, W2q, s2 = moe_w
    x, ids, gw = S.moe_inputs(M, K, TOPK, E, rep=7, device=cuda_device)
    a_ref = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=CC)
    y_ref = dg.dg_moe_w2(a_ref, ids, gw, W2q, s2, choice=CC)
    for wpc in (2, 4, 8):
        for tile in (0, 8, 48, 1536):
            for mt in (0, 1, 2, 4, 8):
                c = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, wpc, 0, tile, mt)
                a = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=c)
                assert torch.equal(a.view(torch.int16), a_ref.view(torch.int16)), (wpc, tile, mt)
                c2 = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, wpc, 0, 4 * tile if tile else 0, mt)
                y = dg.dg_moe_w2(a_ref, ids, gw, W2q, s2, choice=c2)
                assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), (wpc, tile, mt)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_moe_range_order_bitwise_identical_to_units(cuda_device, moe_w, M):
    """The row-range order computes every output with the same canonical chain as the
    (expert, N-tile) order: the same bits for every geometry."""
    W1q, s1, W2q, s2 = moe_w
    x, ids, gw = S.moe_inputs(M, K, TOPK, E, rep=11, device=cuda_device)
    a_ref = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=CC)
    y_ref = dg.dg_moe_w2(a_ref, ids, gw, W2q, s2, choice=CC)
    for wpc in (4, 8):
        for cps in (0, 1, 2, 3):
            for mt in (0, 1, 2, 4, 8):
                c = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, wpc, cps, 0, mt, 2)
                a = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=c)
                assert torch.equal(a.view(torch.int16), a_ref.view(torch.int16)), (wpc, cps, mt)
                y = dg.dg_moe_w2(a_ref, ids, gw, W2q, s2, choice=c)
                assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), (wpc, cps, mt)


@pytest.mark.parametrize("M,E_,I_,K_,Nout,topk", [(1, 8, 80, 272, 100, 3), (3, 8, 80, 272, 100, 3),
                                                  (2, 16, 208, 64, 1000, 5), (7, 4, 16, 16, 9, 2),
                                                  (10, 128, 1536, 4096, 4096, 6)])
def test_moe_range_order_ragged_shapes(cuda_device, M, E_, I_, K_, Nout, topk):
    """Ranges of one row, CTAs with no work, a short last range, column counts that
    leave half a pair: against the (expert, N-tile) order bit for bit and the oracle."""
    W1q, s1, W2q, s2 = S.moe_weights(E_, I_, K_, Nout, device=cuda_device)
    x, ids, gw = S.moe_inputs(M, K_, topk, E_, rep=2, device=cuda_device)
    a = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=RANGE)
    y = dg.dg_moe_w2(a, ids, gw, W2q, s2, choice=RANGE)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=CC).view(torch.int16))
    assert torch.equal(y.view(torch.int16), dg.dg_moe_w2(a, ids, gw, W2q, s2, choice=CC).view(torch.int16))
    if E_ <= 16:
        r = O.moe_w1_silu(bits16(x), ids.cpu().numpy(), W1q.cpu().numpy(), s1.cpu().numpy())
        exc = silu_excess(f64(a), r["g"], r["u"], r["absg"], r["absu"], r["a"])
        assert (exc <= 0).all()
        ref, bound = O.moe_w2(bits16(a), ids.cpu().numpy(), gw.cpu().numpy(), W2q.cpu().numpy(), s2.cpu().numpy())
        assert (lin_excess(f64(y), ref, bound) <= 0).all()


def test_moe_range_order_refuses_what_does_not_fit(cuda_device, moe_w):
    W1q, s1, W2q, s2 = moe_w
    M = RANGE_W2_MAX_M + 1
    x, ids, gw = S.moe_inputs(M, K, TOPK, E, device=cuda_device)
    a = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=RANGE)        # W1 keeps token rows: fits
    with pytest.raises(dg.DGError):
        dg.dg_moe_w2(a, ids, gw, W2q, s2, choice=RANGE)
    for bad in (dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 2, 0, 0, 0, 2),      # 2 warps
                dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 5, 0, 0, 2),      # 5 CTAs per SM
                dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0, 1, 0, 2),      # params[3] must be 0
                dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0, 0, 0, 3)):     # no order 3
        with pytest.raises(dg.DGError):
            dg.dg_moe_w1_silu(x[:1].contiguous(), ids[:1].contiguous(), W1q, s1, choice=bad)


@pytest.mark.parametrize("family", ["cc", "tc", "range"])
def test_moe_invalid_ids_flag_and_zero(cuda_device, moe_w, family):
    W1q, s1, W2q, s2 = moe_w
    c = FAMILIES[family]
    M = 3
    x, ids, gw = S.moe_inputs(M, K, TOPK, E, device=cuda_device)
    bad = ids.clone()
    bad[0, 2] = bad[0, 1]        # repeated expert
    bad[1, 5] = 500              # out of range
    bad[2, 0] = -3
    ws = dg.workspace(dg.DG_OP_MOE_W1, M, I, K, TOPK)
    a = dg.dg_moe_w1_silu(x, bad, W1q, s1, ws=ws, choice=c)
    assert dg.dg_device_status(ws) & 0x1
    assert (a[0, 2] == 0).all() and (a[1, 5] == 0).all() and (a[2, 0] == 0).all()
    dg.dg_device_status_clear(ws)
    assert dg.dg_device_status(ws) == 0
    ws2 = dg.workspace(dg.DG_OP_MOE_W2, M, K, I, TOPK)
    y = dg.dg_moe_w2(a, bad, gw, W2q, s2, ws=ws2, choice=c)
    torch.cuda.synchronize()
    assert dg.dg_device_status(ws2) & 0x1
    # the oracle skips the same slots
    ids_np = bad.cpu().numpy()
    used = np.unique(ids_np[(ids_np >= 0) & (ids_np < E)])
    remap = {int(e): i for i, e in enumerate(used)}
    ids_c = np.array([[remap.get(int(e), -1) for e in row] for row in ids_np], np.int32)
    sel = torch.as_tensor(used, device=cuda_device)
    ref, bound = O.moe_w2(bits16(a), ids_c, gw.cpu().numpy(), W2q[sel].cpu().numpy(), s2[sel].cpu().numpy())
    exc = lin_excess(f64(y), ref, bound)
    assert (exc <= 0).all()


def test_moe_many_pairs_on_one_expert(cuda_device):
    """Every token routes to the same experts: one expert's pairs span several passes."""
    W1q, s1, W2q, s2 = S.moe_weights(8, 64, 256, 128, device=cuda_device)
    M = 16
    x, ids, gw = S.moe_inputs(M, 256, 3, 8, device=cuda_device)
    ids[:] = torch.tensor([5, 2, 7], dtype=torch.int32, device=cuda_device)
    for c in [dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0, 0, mt) for mt in (1, 2, 8)] + [TC]:
        mt = c.params[4]
        a = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=c)
        y = dg.dg_moe_w2(a, ids, gw, W2q, s2, choice=c)
        torch.cuda.synchronize()
        r = O.moe_w1_silu(bits16(x), ids.cpu().numpy(), W1q.cpu().numpy(), s1.cpu().numpy())
        exc = silu_excess(f64(a), r["g"], r["u"], r["absg"], r["absu"], r["a"])
        assert (exc <= 0).all(), mt
        ref, bound = O.moe_w2(bits16(a), ids.cpu().numpy(), gw.cpu().numpy(), W2q.cpu().numpy(), s2.cpu().numpy())
        assert (lin_excess(f64(y), ref, bound) <= 0).all(), mt


@pytest.mark.parametrize("family", ["cc", "tc", "range"])
def test_moe_token_without_valid_slot_gives_zero(cuda_device, family):
    W1q, s1, W2q, s2 = S.moe_weights(8, 64, 256, 128, device=cuda_device)
    x, ids, gw = S.moe_inputs(2, 256, 3, 8, device=cuda_device)
    ids[1] = -1
    a = dg.dg_moe_w1_silu(x, ids, W1q, s1, choice=FAMILIES[family])
    y = dg.dg_moe_w2(a, ids, gw, W2q, s2, choice=FAMILIES[family])
    torch.cuda.synchronize()
    assert (y[1] == 0).all() and (a[1] == 0).all()
    assert (y[0] != 0).any()


@pytest.mark.parametrize("family", ["cc", "tc", "range"])
def test_moe_single_expert_equals_scaled_gemv(cuda_device, family):
    """One token, one slot, gate weight 1: W2 reduces to a per-row-scaled fp8 GEMV."""
    W1q, s1, W2q, s2 = S.moe_weights(4, 512, 1024, 768, device=cuda_device)
    a = torch.randn((1, 1, 512), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16).to(cuda_device)
    ids = torch.tensor([[2]], dtype=torch.int32, device=cuda_device)
    gw = torch.ones((1, 1), dtype=torch.float32, device=cuda_device)
    y = dg.dg_moe_w2(a, ids, gw, W2q, s2, choice=FAMILIES[family])
    torch.cuda.synchronize()
    lg, ad = O.head_fp8(bits16(a[0]), W2q[2].cpu().numpy(), 1.0)
    s = s2[2].cpu().numpy().astype(np.float64)
    exc = lin_excess(f64(y), lg * s, ad * s)
    assert (exc <= 0).all()


@pytest.mark.parametrize("M,E,seed,bad", [(1, 128, 1, False), (2, 128, 2, False), (5, 8, 3, True), (7, 128, 4, True),
                                          (16, 128, 5, False), (16, 16, 6, True), (3, 1000, 7, True)])
def test_moe_routing_tables_match_oracle(cuda_device, M, E, seed, bad):
    """The routing scan the MoE kernels run, exported, equals the oracle's grouping bit for bit."""
    topk = 6
    ids, _ = S.moe_routing(M, topk, E, seed=seed)
    if bad:                                   # repeated and out-of-range ids
        g = torch.Generator().manual_seed(seed)
        for _ in range(max(1, M)):
            t, k = int(torch.randint(M, (1,), generator=g)), int(torch.randint(topk, (1,), generator=g))
            ids[t, k] = [-1, E, E + 7, int(ids[t, 0])][int(torch.randint(4, (1,), generator=g))]
    ws = dg.workspace(dg.DG_OP_MOE_W1, M, 64, 64, topk)
    r = dg.dg_moe_route_debug(ids.to(cuda_device), E, ws=ws)
    ref = O.moe_route(ids.numpy(), E)
    assert np.array_equal(r["valid"], ref["valid"])
    assert np.array_equal(r["nvalid"], ref["valid"].sum(axis=1))
    assert np.array_equal(r["experts"], ref["experts"]) and r["U"] == len(ref["experts"])
    assert np.array_equal(r["offsets"], ref["offsets"]) and r["P"] == int(ref["offsets"][-1])
    assert np.array_equal(r["pair_tok"], ref["pair_tok"])
    assert np.array_equal(r["pair_slot"], ref["pair_slot"])
    assert bool(dg.dg_device_status(ws) & dg.DG_DEVERR_BAD_TOPK_ID) == bool((ref["valid"] == 0).any())


def test_moe_routing_export_rejects_bad_arguments(cuda_device):
    ids = torch.zeros((2, 6), dtype=torch.int32, device=cuda_device)
    for kw in (dict(E=0), dict(E=2000)):
        with pytest.raises(dg.DGError):
            dg.dg_moe_route_debug(ids, **kw)
    with pytest.raises(dg.DGError):
        dg.dg_moe_route_debug(torch.zeros((17, 6), dtype=torch.int32, device=cuda_device), 128)
