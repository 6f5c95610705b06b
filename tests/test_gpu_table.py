"""On-device sweep -> shape table -> selector, on a GPU.

The sweep keeps every candidate's time beside the pick, promotes only bitwise-equal
candidates at least 2 % faster than the default, and a loaded table drives dg_select;
results through an engaged table equal the default's bits.
"""
import json

import pytest
import torch

import gemv_dg_bf16_gb300 as dg
from synth import decode_inputs as S

pytestmark = pytest.mark.gpu

SHAPES = [
    (dg.DG_OP_GEMV_BF16, 1, 2048, 1024, 0, 0),
    (dg.DG_OP_GEMV_BF16, 16, 4096, 1024, 0, 0),
    (dg.DG_OP_GATE_UP_SILU, 2, 1024, 1024, 0, 0),
    (dg.DG_OP_HEAD_FP8_ARGMAX, 1, 8192, 1024, 0, 0),
    (dg.DG_OP_MOE_W1, 2, 256, 512, 6, 16),
    (dg.DG_OP_MOE_W2, 2, 512, 256, 6, 16),
    (dg.DG_OP_GEMV_A8W8, 4, 2048, 1024, 0, 0),
]


@pytest.fixture(scope="module")
def table(tmp_path_factory, cuda_device):
    path = str(tmp_path_factory.mktemp("tab") / "table.json")
    dg.dg_sweep(SHAPES, path, reps=5)
    with open(path) as f:
        return path, json.load(f)


def test_sweep_table_contents(table):
    path, doc = table
    assert doc["format"] == "libdecodegemm-table"
    assert doc["identity"]["selection_space"] == dg.dg_selection_space()
    assert doc["identity"]["build"] == dg.dg_build_id()
    assert len(doc["entries"]) == len(SHAPES)
    for e in doc["entries"]:
        cands = e["candidates"]
        assert len(cands) >= 2                               # every candidate kept beside the pick
        assert all(c["us"] > 0 for c in cands)
        d = [c for c in cands if c["variant"] == e["default"]["variant"] and c["params"] == e["default"]["params"]]
        assert d and d[0]["bitwise"]
        pk = [c for c in cands if c["variant"] == e["pick"]["variant"] and c["params"] == e["pick"]["params"]]
        assert pk and pk[0]["bitwise"]                       # only byte-identical candidates are picked
        if e["pick"] != e["default"]:
            assert e["pick_us"] <= 0.98 * e["default_us"]    # the 2 % promotion floor
        fams = {3 if c["variant"] == 3 else 1 for c in cands}   # CC_WARP and CC_BULK are one family
        assert len(fams) == 1                                # one kernel family per bucket


def test_engaged_table_drives_select_and_keeps_bits(table, cuda_device):
    path, doc = table
    M, N, K = 16, 4096, 1024
    x, W = S.linear_inputs(M, N, K, device=cuda_device)
    ref = dg.dg_gemv_bf16(x, W)                              # compiled default
    dg.dg_table_load(path)
    try:
        assert dg.dg_table_entries() == len(SHAPES)
        c = dg.dg_select(dg.DG_OP_GEMV_BF16, 13, N, K)       # 13 pads up to the 16 bucket
        assert c.from_table == 1
        ent = [e for e in doc["entries"] if e["op"] == "gemv_bf16" and e["M"] == 16][0]
        assert [c.variant, list(c.params)] == [ent["pick"]["variant"], ent["pick"]["params"]]
        y = dg.dg_gemv_bf16(x, W)
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
        assert dg.dg_select(dg.DG_OP_GEMV_BF16, 16, 4096, 4096).from_table == 0   # no nearest-size fallback
    finally:
        dg.dg_table_clear()
    assert dg.dg_table_entries() == 0


def test_stale_table_refused_on_device(table, tmp_path, cuda_device):
    path, doc = table
    doc = dict(doc)
    doc["identity"] = dict(doc["identity"], selection_space=99)
    bad = tmp_path / "stale.json"
    bad.write_text(json.dumps(doc))
    with pytest.raises(dg.DGError) as e:
        dg.dg_table_load(str(bad))
    assert e.value.status == 6
    assert dg.dg_table_entries() == 0


def test_batch_invariant_mode_ignores_picks_of_the_other_family(table, cuda_device):
    """A loaded table's CUDA-core pick (1 row) is not used in the batch-invariant mode;
    a tensor-core pick (16 rows) is, with the K-split fixed by the shape."""
    path, doc = table
    dg.dg_table_load(path)
    try:
        assert dg.dg_select(dg.DG_OP_GEMV_BF16, 1, 2048, 1024).from_table == 1
        dg.dg_set_numerics(dg.DG_NUMERICS_BATCH_INVARIANT)
        try:
            c1 = dg.dg_select(dg.DG_OP_GEMV_BF16, 1, 2048, 1024)
            assert c1.variant == dg.DG_VAR_TC and c1.from_table == 0 and c1.params[1] == 1
            c16 = dg.dg_select(dg.DG_OP_GEMV_BF16, 16, 4096, 1024)
            ent = [e for e in doc["entries"] if e["op"] == "gemv_bf16" and e["M"] == 16][0]
            assert c16.from_table == 1 and c16.variant == ent["pick"]["variant"] == dg.DG_VAR_TC
            assert c16.params[0] == ent["pick"]["params"][0] and c16.params[1] == 1
            # the two rows computed through the mode agree with a 16-row call
            x, W = S.linear_inputs(16, 4096, 1024, device=cuda_device)
            y16 = dg.dg_gemv_bf16(x, W)
            y1 = dg.dg_gemv_bf16(x[:1].contiguous(), W)
            assert torch.equal(y1.view(torch.int16), y16[:1].view(torch.int16))
        finally:
            dg.dg_set_numerics(dg.DG_NUMERICS_FASTEST)
    finally:
        dg.dg_table_clear()


def test_sweep_resumes_a_partial_table(tmp_path, cuda_device):
    """An interrupted sweep (here: only the first half of the shapes written) continues
    where it stopped: the finished entries stay as they are, the rest are measured."""
    path = str(tmp_path / "partial.json")
    half = SHAPES[:3]
    dg.dg_sweep(half, path, reps=3)
    with open(path) as f:
        first = json.load(f)
    dg.dg_sweep(SHAPES, path, reps=3, resume=True)
    with open(path) as f:
        done = json.load(f)
    assert len(done["entries"]) == len(SHAPES)
    assert done["entries"][:3] == first["entries"]
    assert done["identity"] == first["identity"]
    dg.dg_table_load(path)                       # the merged table passes the identity checks
    try:
        assert dg.dg_table_entries() == len(SHAPES)
    finally:
        dg.dg_table_clear()
    before = open(path).read()
    dg.dg_sweep(SHAPES, path, reps=3, resume=True)    # nothing left to measure
    assert open(path).read() == before
