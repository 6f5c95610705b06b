"""Host-side checks of the C ABI that need no GPU: exports, argument errors, the shape
table parser and its refusals, bucket padding and the dispatch knob."""
import ctypes
import json
import os
import subprocess
import sys

import pytest

import gemv_dg_bf16_gb300 as dg
from gemv_dg_bf16_gb300 import _binding as B
from tests._helpers import ROOT, header_functions


@pytest.fixture(scope="module", autouse=True)
def built():
    from gemv_dg_bf16_gb300 import build
    build.build()
    return dg.lib()


def test_library_exports_every_declared_function():
    names = header_functions()
    assert len(names) >= 18
    L = ctypes.CDLL(dg.library_path())
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_library_has_no_oracle_dependency():
    out = subprocess.run(["nm", "-D", dg.library_path()], capture_output=True, text=True).stdout
    assert "dgo_" not in out


def test_rows_buckets_one_list():
    assert dg.ROWS_BUCKETS == (1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128, 192, 256, 384, 512)


def test_status_strings():
    assert dg.dg_status_str(0) == "ok"
    assert "aligned" in dg.dg_status_str(2)
    assert dg.dg_status_str(99) == "unknown status"


# Fake device addresses: every call below fails an argument check before any launch.
A = 0x10000            # 16-byte aligned
U = 0x10002            # misaligned


def _gemv(x=A, W=A, y=A, M=2, N=64, K=256, ws=A, wsb=4096):
    return dg.lib().dg_gemv_bf16(ctypes.c_void_p(x), ctypes.c_void_p(W), ctypes.c_void_p(y), M, N, K,
                                 ctypes.c_void_p(ws), wsb, None, None)


def test_argument_errors_before_any_device_work():
    assert _gemv(M=0) == 1
    assert _gemv(M=513) == 1
    assert _gemv(K=250) == 3
    assert _gemv(x=0) == 1
    assert _gemv(W=U) == 2
    assert _gemv(ws=U) == 2
    assert _gemv(wsb=8) == 4
    L = dg.lib()
    P = ctypes.c_void_p
    assert L.dg_head_fp8_argmax(P(A), P(A), None, P(A), P(A), 2, 100, 64, P(A), 1 << 20, None, None) == 1
    assert L.dg_head_fp8_argmax(P(A), P(A), P(A), P(A), P(A), 9, 100, 64, P(A), 1 << 20, None, None) == 1
    assert L.dg_head_fp8_argmax(P(A), P(A), P(A), P(A), P(A), 2, 100, 40, P(A), 1 << 20, None, None) == 3
    assert L.dg_head_fp8_argmax(P(A), P(A), P(A), P(U), P(A), 2, 100, 64, P(A), 1 << 20, None, None) == 2
    assert L.dg_moe_w1_silu(P(A), P(A), P(A), P(A), P(A), 17, 6, 128, 1536, 4096, P(A), 1 << 20, None, None) == 1
    assert L.dg_moe_w1_silu(P(A), P(A), P(A), P(A), P(A), 2, 9, 128, 1536, 4096, P(A), 1 << 20, None, None) == 1
    assert L.dg_moe_w2(P(A), P(A), P(A), P(A), P(A), P(A), 2, 6, 128, 1544, 4096, P(A), 1 << 24, None, None) == 3
    assert L.dg_moe_w2(P(A), P(A), P(A), P(A), P(A), P(A), 2, 6, 128, 1536, 4096, P(A), 64, None, None) == 4


def test_workspace_sizes():
    assert dg.dg_workspace_bytes(dg.DG_OP_GEMV_BF16, 1, 4096, 4096) >= 16
    assert dg.dg_workspace_bytes(dg.DG_OP_HEAD_FP8_ARGMAX, 8, 248320, 4096) >= 256 + 4096 * 8 * 8
    w2 = dg.dg_workspace_bytes(dg.DG_OP_MOE_W2, 16, 4096, 1536, 6)
    assert w2 >= 16 * 6 * 4096 * 4


def test_select_defaults_and_bucket_padding():
    for op in range(5):
        for M in (1, 5, 7, 100, 128):
            if op == dg.DG_OP_HEAD_FP8_ARGMAX and M > 8 or op >= dg.DG_OP_MOE_W1 and M > 16:
                continue
            c = dg.dg_select(op, M, 4096, 4096)
            dense_bf16 = op in (dg.DG_OP_GEMV_BF16, dg.DG_OP_GATE_UP_SILU)
            head = op == dg.DG_OP_HEAD_FP8_ARGMAX
            w1 = op == dg.DG_OP_MOE_W1
            w2 = op == dg.DG_OP_MOE_W2
            # buckets: M=5 -> 6, M=7 -> 8
            want = dg.DG_VAR_TC if ((dense_bf16 and M >= 13) or (head and M >= 2) or (w1 and M >= 7)
                                    or (w2 and M >= 5)) else dg.DG_VAR_CC_WARP
            # the warp-level tensor cores take the linear at 2-12 rows and gate/up at 3-8
            if dense_bf16 and ((2 <= M <= 12) if op == dg.DG_OP_GEMV_BF16 else (3 <= M <= 8)):
                want = dg.DG_VAR_MMA
            assert c.variant == want and c.from_table == 0, (op, M, c)
    assert dg.dg_select(0, 129, 4096, 4096).variant == dg.DG_VAR_TC     # mid-M bucket 192
    # MoE: the row-range order (params[5] = 2) at 1-2 rows (W1) and 1-4 rows (W2), the
    # (expert, N-tile) order for W1 at 3-6 rows, the tensor cores above
    order = lambda op, M: dg.dg_select(op, M, 1536 if op == dg.DG_OP_MOE_W1 else 4096,
                                       4096 if op == dg.DG_OP_MOE_W1 else 1536).params[5]
    assert [order(dg.DG_OP_MOE_W1, M) for M in (1, 2, 3, 6)] == [2, 2, 0, 0]
    assert [order(dg.DG_OP_MOE_W2, M) for M in (1, 2, 3, 4)] == [2, 2, 2, 2]
    assert dg.dg_select(dg.DG_OP_MOE_W2, 5, 4096, 1536).variant == dg.DG_VAR_TC
    with pytest.raises(dg.DGError):
        dg.dg_select(0, 513, 4096, 4096)
    # a bucket's default does not depend on where in the bucket M falls
    assert dg.dg_select(0, 5, 64, 64).as_tuple() == dg.dg_select(0, 6, 64, 64).as_tuple()


# ---------------------------------------------------------------- shape table

ARCH, DRV, RT = "sm_103", 13000, 13000


def _table(tmp_path, **over):
    ident = {"arch": ARCH, "driver": DRV, "runtime": RT, "build": dg.dg_build_id(),
             "selection_space": dg.dg_selection_space()}
    ident.update(over.pop("identity", {}))
    for k in over.pop("drop", []):
        ident.pop(k)
    entries = over.pop("entries", [
        {"op": "gemv_bf16", "M": 1, "N": 4096, "K": 4096,
         "pick": {"variant": 1, "params": [2, 4, 0, 0, 0, 0]}, "pick_us": 5.0,
         "default": {"variant": 1, "params": [4, 8, 0, 0, 0, 0]}, "default_us": 5.2,
         "candidates": [{"variant": 1, "params": [4, 8, 0, 0, 0, 0], "us": 5.2, "bitwise": True},
                        {"variant": 1, "params": [2, 4, 0, 0, 0, 0], "us": 5.0, "bitwise": True}]},
        {"op": "moe_w2", "M": 16, "N": 4096, "K": 1536,
         "pick": {"variant": 1, "params": [4, 8, 0, 64, 0, 0]}, "pick_us": 50.0}])
    doc = {"format": "libdecodegemm-table", "identity": ident, "entries": entries}
    doc.update(over)
    p = tmp_path / "table.json"
    p.write_text(json.dumps(doc))
    return str(p)


def _check(path, **kw):
    return dg.dg_table_check(path, kw.get("arch", ARCH), kw.get("drv", DRV), kw.get("rt", RT))


def test_table_valid(tmp_path):
    s, n, why = _check(_table(tmp_path))
    assert (s, n) == (0, 2), why


@pytest.mark.parametrize("kw,needle", [
    (dict(drop=["selection_space"]), "made before the kernel selection space"),
    (dict(identity={"selection_space": 99}), "selection space 99"),
    (dict(identity={"arch": "sm_100"}), "architecture sm_100"),
    (dict(identity={"driver": 12080}), "driver 12080"),
    (dict(identity={"runtime": 1}), "runtime 1"),
    (dict(identity={"build": "0123"}), "library build 0123"),
    (dict(entries=[{"op": "gemv_bf16", "M": 5, "N": 1, "K": 8, "pick": {"variant": 1, "params": [4, 8]}}]),
     "not a decode bucket"),
    (dict(entries=[{"op": "gemv_bf16", "M": 4, "N": 1, "K": 8, "pick": {"variant": 7, "params": [4, 8]}}]),
     "selection space"),
    (dict(entries=[{"op": "gate_up_silu", "M": 4, "N": 1, "K": 8, "pick": {"variant": 1, "params": [1, 8]}}]),
     "even"),
    (dict(entries=[{"op": "nope", "M": 4, "N": 1, "K": 8, "pick": {"variant": 1, "params": [4, 8]}}]),
     "unknown op"),
    (dict(entries=[{"op": "gemv_bf16", "M": 1, "N": 1, "K": 8, "pick": {"variant": 1, "params": [4, 4, 0, 3]}}]),
     "K-split warps must be 1, 2, 4 or 8"),
    (dict(entries=[{"op": "gemv_bf16", "M": 1, "N": 1, "K": 8, "pick": {"variant": 1, "params": [4, 2, 0, 4]}}]),
     "divide warps per CTA"),
    (dict(entries=[{"op": "gemv_bf16", "M": 4, "N": 1, "K": 8}]), "pick"),
    (dict(format="other"), "not a libdecodegemm table"),
])
def test_table_refusals(tmp_path, kw, needle):
    s, n, why = _check(_table(tmp_path, **kw))
    assert s == 6 and n == 0 and needle in why, why


def test_table_corrupt_and_truncated(tmp_path):
    good = _table(tmp_path)
    text = open(good).read()
    bad = tmp_path / "trunc.json"
    bad.write_text(text[: len(text) // 2])
    s, _, why = _check(str(bad))
    assert s == 6 and "not a valid table" in why
    s, _, why = _check(str(tmp_path / "missing.json"))
    assert s == 6 and "cannot read" in why
    garbage = tmp_path / "garbage.json"
    garbage.write_bytes(b"\x00\xff{{{")
    assert _check(str(garbage))[0] == 6


def test_table_refused_when_dispatch_knob_set(tmp_path):
    path = _table(tmp_path)
    code = ("import sys; sys.path.insert(0, %r); import gemv_dg_bf16_gb300 as dg; "
            "s, n, why = dg.dg_table_check(%r, 'sm_103', 13000, 13000); print(s, why)") % (ROOT, path)
    env = dict(os.environ, DG_FORCE_VARIANT="1:2,4,0,0")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True).stdout
    assert out.startswith("6 ") and "DG_FORCE_VARIANT" in out


def test_force_knob_drives_select():
    code = ("import sys; sys.path.insert(0, %r); import gemv_dg_bf16_gb300 as dg; "
            "c = dg.dg_select(0, 3, 64, 64); print(c.variant, list(c.params))") % ROOT
    env = dict(os.environ, DG_FORCE_VARIANT="1:2,4,1,0")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True).stdout
    assert out.split() [:3] == ["1", "[2,", "4,"]
    env = dict(os.environ, DG_FORCE_VARIANT="5:1,1,0,0")
    code_bad = code.replace("c = dg.dg_select(0, 3, 64, 64); print(c.variant, list(c.params))",
                            "print(dg.lib().dg_select(0, 3, 64, 64, dg._binding.ctypes.byref(dg.Choice())))")
    out = subprocess.run([sys.executable, "-c", code_bad], env=env, capture_output=True, text=True, check=True).stdout
    assert out.strip() == "8"


def test_binding_constants_match_header():
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dg.h")).read()
    enums = dict((k, int(v)) for k, v in re.findall(r"\b(DG_(?:OK|ERR_\w+))\s*=\s*(\d+)", hdr))
    defines = dict((k, int(v, 16)) for k, v in re.findall(r"#define\s+(DG_DEVERR_\w+)\s+0x([0-9A-Fa-f]+)", hdr))
    assert len(enums) == 9 and len(defines) == 2
    for name, val in {**enums, **defines}.items():
        assert getattr(dg, name) == val, name


def test_batch_invariant_numerics_takes_one_family_per_op():
    assert dg.dg_numerics() == dg.DG_NUMERICS_FASTEST
    with pytest.raises(dg.DGError):
        dg.dg_set_numerics(2)
    # the fastest mode mixes families across row buckets
    assert dg.dg_select(dg.DG_OP_GEMV_BF16, 1, 4096, 4096).variant == dg.DG_VAR_CC_WARP
    assert dg.dg_select(dg.DG_OP_GEMV_BF16, 8, 4096, 4096).variant == dg.DG_VAR_MMA
    assert dg.dg_select(dg.DG_OP_GEMV_BF16, 16, 4096, 4096).variant == dg.DG_VAR_TC
    dg.dg_set_numerics(dg.DG_NUMERICS_BATCH_INVARIANT)
    try:
        assert dg.dg_numerics() == dg.DG_NUMERICS_BATCH_INVARIANT
        top = {dg.DG_OP_GEMV_BF16: 512, dg.DG_OP_GATE_UP_SILU: 512, dg.DG_OP_HEAD_FP8_ARGMAX: 8,
               dg.DG_OP_MOE_W1: 16, dg.DG_OP_MOE_W2: 16}
        for op, mmax in top.items():
            picks = {dg.dg_select(op, M, 4096, 4096).as_tuple() for M in range(1, mmax + 1)}
            assert {p[0] for p in picks} == {dg.DG_VAR_TC}, (op, picks)
            dense = op in (dg.DG_OP_GEMV_BF16, dg.DG_OP_GATE_UP_SILU)
            # the tensor-core linears take the K-split fixed by the shape alone
            assert {p[1][1] for p in picks} == ({1} if dense else {0}), (op, picks)
        # a head too wide for the tensor-core split stays on the CUDA cores at every M
        assert {dg.dg_select(dg.DG_OP_HEAD_FP8_ARGMAX, M, 248320, 16384).variant for M in range(1, 9)} == \
            {dg.DG_VAR_CC_WARP}
    finally:
        dg.dg_set_numerics(dg.DG_NUMERICS_FASTEST)
    assert dg.dg_select(dg.DG_OP_GEMV_BF16, 1, 4096, 4096).variant == dg.DG_VAR_CC_WARP
    assert dg.dg_select(dg.DG_OP_GEMV_BF16, 300, 4096, 4096).params[1] == 0


def test_tc_split_rule_parameter_checked(tmp_path):
    ent = lambda op, p: [{"op": op, "M": 4, "N": 64, "K": 64, "pick": {"variant": 3, "params": p}}]
    assert _check(_table(tmp_path, entries=ent("gemv_bf16", [0, 1])))[0] == 0
    s, _, why = _check(_table(tmp_path, entries=ent("gemv_bf16", [0, 2])))
    assert s == 6 and "K-split rule" in why
    s, _, why = _check(_table(tmp_path, entries=ent("moe_w1_silu", [0, 1])))
    assert s == 6 and "unused tensor-core parameter" in why


def test_moe_work_order_parameters_checked(tmp_path):
    ent = lambda p: [{"op": "moe_w2", "M": 2, "N": 4096, "K": 1536, "pick": {"variant": 1, "params": p}}]
    for ok in ([4, 8, 0, 64, 2, 0], [4, 8, 0, 64, 2, 1], [4, 8, 2, 0, 4, 2], [4, 4, 0, 0, 0, 2]):
        assert _check(_table(tmp_path, entries=ent(ok)))[0] == 0, ok
    for bad, why in (([4, 8, 0, 0, 0, 3], "work order"), ([4, 2, 0, 0, 0, 2], "row-range"),
                     ([4, 8, 5, 0, 0, 2], "row-range"), ([4, 8, 0, 1, 0, 2], "row-range")):
        s, _, reason = _check(_table(tmp_path, entries=ent(bad)))
        assert s == 6 and why in reason, (bad, reason)


def test_a8w8_select_and_argument_errors():
    for M in (1, 2, 5, 16, 33, 64):
        c = dg.dg_select(dg.DG_OP_GEMV_A8W8, M, 8192, 4096)
        assert c.variant == dg.DG_VAR_TC and c.from_table == 0
    assert dg.dg_workspace_bytes(dg.DG_OP_GEMV_A8W8, 64, 8192, 4096) >= 16
    L = dg.lib()
    P = ctypes.c_void_p
    call = lambda x=A, W=A, s=A, y=A, M=2, N=64, K=256, ws=A, wsb=1 << 16, c=None: L.dg_gemv_a8w8_blockscale(
        P(x), P(W), P(s), P(y), M, N, K, P(ws), wsb, None, c)
    assert call(M=0) == 1 and call(M=65) == 1 and call(N=0) == 1
    assert call(K=264) == 3                       # K % 16
    assert call(s=0) == 1 and call(s=U) == 2 and call(W=U) == 2
    assert call(wsb=8) == 4
    bad = dg.Choice.make(dg.DG_VAR_CC_WARP, 4, 8, 0)
    assert dg.lib().dg_quant_a8_blockscale(P(A), P(A), P(A), 2, 40, None) == 3
    assert dg.lib().dg_quant_a8_blockscale(P(A), P(U), P(A), 2, 64, None) == 2
    assert dg.lib().dg_quant_a8_blockscale(None, P(A), P(A), 2, 64, None) == 1


def test_a8w8_table_refuses_cuda_core_pick(tmp_path):
    ent = [{"op": "gemv_a8w8", "M": 4, "N": 64, "K": 64, "pick": {"variant": 1, "params": [4, 8]}}]
    s, _, why = _check(_table(tmp_path, entries=ent))
    assert s == 6 and "tensor cores only" in why
    ent = [{"op": "gemv_a8w8", "M": 4, "N": 64, "K": 64, "pick": {"variant": 3, "params": [4]}}]
    assert _check(_table(tmp_path, entries=ent))[0] == 0


def test_binding_refuses_mismatched_tensors_before_any_call():
    """The C entry points see raw pointers only; the binding checks dtypes and shapes
    first (these CPU tensors never reach the library)."""
    import torch
    bf, u8, f32, i32 = torch.bfloat16, torch.uint8, torch.float32, torch.int32
    x = torch.zeros((2, 256), dtype=bf)
    cases = [
        (lambda: dg.dg_gemv_bf16(x, torch.zeros((64, 128), dtype=bf)), "W: shape"),
        (lambda: dg.dg_gemv_bf16(x, torch.zeros((64, 256), dtype=torch.float16)), "W: dtype"),
        (lambda: dg.dg_gemv_bf16(x, torch.zeros((64, 256), dtype=bf), y=torch.zeros((2, 63), dtype=bf)), "y: shape"),
        (lambda: dg.dg_gate_up_silu(x, torch.zeros((63, 256), dtype=bf)), "W_gu: shape"),
        (lambda: dg.dg_head_fp8_argmax(x, torch.zeros((100, 256), dtype=u8), torch.zeros(1, dtype=torch.float64)),
         "scale: dtype"),
        (lambda: dg.dg_head_fp8_argmax(x, torch.zeros((100, 256), dtype=u8), torch.zeros(1, dtype=f32),
                                       argmax=torch.zeros(2, dtype=torch.int64)), "argmax: dtype"),
        (lambda: dg.dg_moe_w1_silu(x, torch.zeros((2, 6), dtype=torch.int64), torch.zeros((8, 128, 256), dtype=u8),
                                   torch.zeros((8, 128), dtype=f32)), "topk_ids: dtype"),
        (lambda: dg.dg_moe_w1_silu(x, torch.zeros((2, 6), dtype=i32), torch.zeros((8, 128, 256), dtype=u8),
                                   torch.zeros((8, 64), dtype=f32)), "s1: shape"),
        (lambda: dg.dg_moe_w2(torch.zeros((2, 6, 64), dtype=bf), torch.zeros((2, 6), dtype=i32),
                              torch.zeros((2, 5), dtype=f32), torch.zeros((8, 128, 64), dtype=u8),
                              torch.zeros((8, 128), dtype=f32)), "topk_w: shape"),
        (lambda: dg.dg_gemv_a8w8_blockscale(x, torch.zeros((300, 256), dtype=u8), torch.zeros((2, 2), dtype=f32)),
         "sw: shape"),
        (lambda: dg.dg_quant_a8_blockscale(x, sx=torch.zeros((2, 3), dtype=f32)), "sx: shape"),
    ]
    for fn, needle in cases:
        with pytest.raises(ValueError) as e:
            fn()
        assert needle in str(e.value), (needle, str(e.value))


def test_binding_op_variant_and_mode_constants_match_header():
    import re
    hdr = open(os.path.join(ROOT, "include", "dg.h")).read()
    enums = dict((k, int(v)) for k, v in re.findall(r"\b(DG_(?:OP|VAR)_\w+)\s*=\s*(\d+)", hdr))
    defines = dict((k, int(v, 0)) for k, v in re.findall(r"#define\s+(DG_(?:NUMERICS|LAUNCH)_\w+)\s+(0x[0-9A-Fa-f]+|\d+)", hdr))
    assert {"DG_OP_GEMV_A8W8", "DG_OP_COUNT", "DG_VAR_TC"} <= set(enums)
    assert {"DG_NUMERICS_FASTEST", "DG_NUMERICS_BATCH_INVARIANT", "DG_LAUNCH_PDL"} <= set(defines)
    for name, val in {**enums, **defines}.items():
        if name == "DG_OP_COUNT":
            continue
        assert getattr(dg, name) == val, name


def test_sweep_resume_keys_and_merge():
    """Resuming a sweep measures only the (op, row bucket, N, K) keys a partial table
    lacks, and the merge keeps the old entries beside the new ones."""
    from gemv_dg_bf16_gb300 import _binding as Bd
    old = {"format": "libdecodegemm-table", "identity": {"build": "b1"},
           "entries": [{"op": "gemv_bf16", "M": 16, "N": 4096, "K": 1024, "pick_us": 5.0},
                       {"op": "moe_w2", "M": 2, "N": 512, "K": 256, "pick_us": 9.0}]}
    shapes = [(dg.DG_OP_GEMV_BF16, 13, 4096, 1024, 0, 0),      # bucket 16: already there
              (dg.DG_OP_GEMV_BF16, 17, 4096, 1024, 0, 0),      # bucket 24: missing
              (dg.DG_OP_MOE_W2, 2, 512, 256, 6, 16),           # there
              (dg.DG_OP_GEMV_A8W8, 300, 2048, 1024, 0, 0)]     # bucket 384: missing
    todo = Bd._sweep_remaining(shapes, old)
    assert todo == [shapes[1], shapes[3]]
    new = {"format": "libdecodegemm-table", "identity": {"build": "b1"},
           "entries": [{"op": "gemv_bf16", "M": 24, "N": 4096, "K": 1024, "pick_us": 6.0},
                       {"op": "moe_w2", "M": 2, "N": 512, "K": 256, "pick_us": 8.0}]}
    m = Bd._merge_tables(old, new)
    keys = [(e["op"], e["M"], e["pick_us"]) for e in m["entries"]]
    assert keys == [("gemv_bf16", 16, 5.0), ("gemv_bf16", 24, 6.0), ("moe_w2", 2, 8.0)]
    assert m["identity"] == new["identity"] and Bd._bucket(513) == -1


def test_table_accepts_mid_m_buckets_only(tmp_path):
    ent = lambda M: [{"op": "gemv_bf16", "M": M, "N": 4096, "K": 1024, "pick": {"variant": 3, "params": [4]}}]
    for M in (192, 256, 384, 512):
        assert _check(_table(tmp_path, entries=ent(M)))[0] == 0, M
    for M in (200, 513, 1024):
        s, _, why = _check(_table(tmp_path, entries=ent(M)))
        assert s == 6 and "not a decode bucket" in why, (M, why)


def test_select_pads_every_row_count_to_its_bucket():
    """Every M maps to the default of its bucket (the smallest listed bucket >= M)."""
    for M in range(1, 513):
        b = next(r for r in dg.ROWS_BUCKETS if r >= M)
        assert dg.dg_select(dg.DG_OP_GEMV_BF16, M, 4096, 4096).as_tuple() == \
            dg.dg_select(dg.DG_OP_GEMV_BF16, b, 4096, 4096).as_tuple(), M
