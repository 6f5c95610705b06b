"""ctypes marshalling for libdecodegemm.so.

Tensors are torch tensors on the current CUDA device; their data pointers, the
current stream and plain integers are passed through unchanged.  bf16 tensors
are torch.bfloat16, e4m3 tensors are torch.uint8 (or float8_e4m3fn) codes.
"""
from __future__ import annotations

import ctypes
import json
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBPATH = os.path.join(_HERE, "libdecodegemm.so")

DG_OP_GEMV_BF16, DG_OP_GATE_UP_SILU, DG_OP_HEAD_FP8_ARGMAX, DG_OP_MOE_W1, DG_OP_MOE_W2, DG_OP_GEMV_A8W8 = range(6)
DG_VAR_DEFAULT, DG_VAR_CC_WARP, DG_VAR_CC_BULK, DG_VAR_TC, DG_VAR_MMA = range(5)
(DG_OK, DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT, DG_ERR_UNSUPPORTED_SHAPE, DG_ERR_WORKSPACE_TOO_SMALL, DG_ERR_CUDA,
 DG_ERR_TABLE_REFUSED, DG_ERR_NO_DEVICE, DG_ERR_BAD_VARIANT) = range(9)
DG_DEVERR_BAD_TOPK_ID = 0x1
DG_DEVERR_WAIT_TIMEOUT = 0x2


def _rows_buckets():
    with open(os.path.join(_HERE, "csrc", "dg_rows.h")) as f:
        text = f.read().replace("\\\n", " ")          # the macro continues over several lines
        m = re.search(r"#define DG_ROWS_BUCKETS\(X\)\s+(.*)", text)
    return tuple(int(v) for v in re.findall(r"X\((\d+)\)", m.group(1)))


ROWS_BUCKETS = _rows_buckets()


class Choice(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("params", ctypes.c_int32 * 6),
                ("from_table", ctypes.c_int32), ("table_us", ctypes.c_float)]

    @classmethod
    def make(cls, variant: int, *params: int) -> "Choice":
        c = cls()
        c.variant = variant
        for i, p in enumerate(params):
            c.params[i] = p
        return c

    def as_tuple(self):
        return (self.variant, tuple(self.params))

    def __repr__(self):
        return f"Choice(variant={self.variant}, params={list(self.params)}, from_table={self.from_table})"


class Shape(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("M", ctypes.c_int32), ("N", ctypes.c_int32),
                ("K", ctypes.c_int32), ("topk", ctypes.c_int32), ("E", ctypes.c_int32)]


class DGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dg_status_str(status)} (status {status})")


_lib = None


def library_path() -> str:
    return _LIBPATH


def lib():
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIBPATH):
        raise ImportError(f"libdecodegemm.so is not built at {_LIBPATH}; run __graft_entry__.build()")
    L = ctypes.CDLL(_LIBPATH)
    P, I, Z, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int
    L.dg_init.argtypes = [I]
    L.dg_status_str.argtypes = [S]
    L.dg_status_str.restype = ctypes.c_char_p
    L.dg_workspace_bytes.argtypes = [I, I, I, I, I]
    L.dg_workspace_bytes.restype = Z
    L.dg_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32), P]
    L.dg_device_status_clear.argtypes = [P, P]
    L.dg_selftest_wait_timeout.argtypes = [P, I, P]
    L.dg_selftest_wait_timeout.restype = S
    L.dg_moe_route_debug.argtypes = [P, I, I, I, P, P, P]
    L.dg_moe_route_debug.restype = S
    L.dg_set_launch_flags.argtypes = [ctypes.c_uint]
    L.dg_set_launch_flags.restype = S
    L.dg_launch_flags.argtypes = []
    L.dg_launch_flags.restype = ctypes.c_uint
    L.dg_set_numerics.argtypes = [I]
    L.dg_set_numerics.restype = S
    L.dg_numerics.argtypes = []
    L.dg_numerics.restype = I
    L.dg_gemv_bf16.argtypes = [P, P, P, I, I, I, P, Z, P, P]
    L.dg_gate_up_silu.argtypes = [P, P, P, I, I, I, P, Z, P, P]
    L.dg_head_fp8_argmax.argtypes = [P, P, P, P, P, I, I, I, P, Z, P, P]
    L.dg_head_fp8_argmax_noalloc.argtypes = [P, P, P, P, P, I, I, I, P, P]
    L.dg_head_fp8_argmax_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int32), P]
    L.dg_head_fp8_argmax_noalloc_scratch.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    L.dg_moe_w1_silu.argtypes = [P, P, P, P, P, I, I, I, I, I, P, Z, P, P]
    L.dg_moe_w2.argtypes = [P, P, P, P, P, P, I, I, I, I, I, P, Z, P, P]
    L.dg_gemv_a8w8_blockscale.argtypes = [P, P, P, P, I, I, I, P, Z, P, P]
    L.dg_quant_a8_blockscale.argtypes = [P, P, P, I, I, P]
    L.dg_select.argtypes = [I, I, I, I, ctypes.POINTER(Choice)]
    L.dg_table_load.argtypes = [ctypes.c_char_p]
    L.dg_table_clear.argtypes = []
    L.dg_table_clear.restype = None
    L.dg_table_entries.argtypes = []
    L.dg_selection_space.argtypes = []
    L.dg_build_id.argtypes = []
    L.dg_build_id.restype = ctypes.c_char_p
    L.dg_table_check.argtypes = [ctypes.c_char_p, ctypes.c_char_p, I, I, ctypes.POINTER(ctypes.c_int),
                                 ctypes.c_char_p, Z]
    L.dg_sweep.argtypes = [ctypes.POINTER(Shape), I, ctypes.c_char_p, I]
    for name in ("dg_init", "dg_device_status", "dg_device_status_clear", "dg_gemv_bf16",
                 "dg_gate_up_silu", "dg_head_fp8_argmax", "dg_head_fp8_argmax_noalloc",
                 "dg_head_fp8_argmax_noalloc_status", "dg_head_fp8_argmax_noalloc_scratch", "dg_moe_w1_silu",
                 "dg_moe_w2", "dg_select",
                 "dg_gemv_a8w8_blockscale", "dg_quant_a8_blockscale",
                 "dg_table_load", "dg_table_check", "dg_sweep"):
        getattr(L, name).restype = S
    _lib = L
    return L


def dg_status_str(status: int) -> str:
    return lib().dg_status_str(int(status)).decode()


def _ok(status: int, where: str):
    if status != 0:
        raise DGError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _choice(choice):
    if choice is None:
        return None
    if isinstance(choice, Choice):
        return ctypes.byref(choice)
    return ctypes.byref(Choice.make(*choice))


_FP8 = tuple(d for d in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if d is not None)


def _expect(t, name, dtypes, shape=None, min_numel=None):
    """Dtype and shape of a tensor argument.  The C entry points take raw pointers and
    cannot see sizes, so a mismatch is refused here (ValueError) before any call."""
    if t is None:
        return
    dtypes = dtypes if isinstance(dtypes, tuple) else (dtypes,)
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {' or '.join(str(d) for d in dtypes)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected at least {min_numel}")


def _nbytes(t):
    return t.numel() * t.element_size()


def _check_dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def dg_init(device: int = 0):
    _ok(lib().dg_init(int(device)), "dg_init")


DG_LAUNCH_PDL = 0x1


def dg_set_launch_flags(flags: int):
    _ok(lib().dg_set_launch_flags(int(flags)), "dg_set_launch_flags")


def dg_launch_flags() -> int:
    return int(lib().dg_launch_flags())


DG_NUMERICS_FASTEST = 0
DG_NUMERICS_BATCH_INVARIANT = 1


def dg_set_numerics(mode: int):
    _ok(lib().dg_set_numerics(int(mode)), "dg_set_numerics")


def dg_numerics() -> int:
    return int(lib().dg_numerics())


def dg_selftest_wait_timeout(ws, timeout_us: int = 20000, stream=None):
    _ok(lib().dg_selftest_wait_timeout(_ptr(ws), int(timeout_us), _stream(stream)), "dg_selftest_wait_timeout")


DG_ROUTE_DEBUG_INTS = 2 + 128 + 16 + 128 + 129 + 128 + 128


def dg_moe_route_debug(topk_ids, E: int, ws=None, stream=None) -> dict:
    """The MoE kernels' routing tables for topk_ids [M, topk] (device int32), as numpy."""
    _expect(topk_ids, "topk_ids", torch.int32)
    _check_dev(topk_ids)
    M, topk = topk_ids.shape
    out = torch.empty(DG_ROUTE_DEBUG_INTS, dtype=torch.int32, device=topk_ids.device)
    if ws is None:
        ws = torch.zeros(256, dtype=torch.uint8, device=topk_ids.device)
    _ok(lib().dg_moe_route_debug(_ptr(topk_ids), M, topk, int(E), _ptr(out), _ptr(ws), _stream(stream)),
        "dg_moe_route_debug")
    o = out.cpu().numpy()
    U, P = int(o[0]), int(o[1])
    valid = o[2:2 + 128]
    nvalid = o[130:146]
    experts = o[146:274]
    offs = o[274:403]
    ptok = o[403:531]
    pslot = o[531:659]
    return dict(U=U, P=P, valid=valid[:M * topk].reshape(M, topk).copy(), nvalid=nvalid[:M].copy(),
                experts=experts[:U].copy(), offsets=offs[:U + 1].copy(), pair_tok=ptok[:P].copy(),
                pair_slot=pslot[:P].copy())


def dg_workspace_bytes(op: int, M: int, N: int, K: int, topk: int = 0) -> int:
    return int(lib().dg_workspace_bytes(op, M, N, K, topk))


def workspace(op: int, M: int, N: int, K: int, topk: int = 0, device=None) -> torch.Tensor:
    """A zero-filled device workspace large enough for (op, M, N, K, topk)."""
    n = dg_workspace_bytes(op, M, N, K, topk)
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def dg_device_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int32(0)
    _ok(lib().dg_device_status(_ptr(ws), ctypes.byref(out), _stream(stream)), "dg_device_status")
    return int(out.value)


def dg_device_status_clear(ws: torch.Tensor, stream=None):
    _ok(lib().dg_device_status_clear(_ptr(ws), _stream(stream)), "dg_device_status_clear")


def dg_gemv_bf16(x, W, y=None, ws=None, choice=None, stream=None):
    """y[M,N] = x[M,K] . W[N,K]^T (bf16 in/out, fp32 accumulation)."""
    M, K = x.shape
    N = W.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(DG_OP_GEMV_BF16, M, N, K, device=x.device)
    _expect(x, "x", torch.bfloat16)
    _expect(W, "W", torch.bfloat16, (N, K))
    _expect(y, "y", torch.bfloat16, (M, N))
    _check_dev(x, W, y, ws)
    _ok(lib().dg_gemv_bf16(_ptr(x), _ptr(W), _ptr(y), M, N, K, _ptr(ws), _nbytes(ws), _stream(stream),
                           _choice(choice)), "dg_gemv_bf16")
    return y


def dg_gemv_a8w8_blockscale(x, Wq, sw, y=None, ws=None, choice=None, stream=None):
    """y[M,N] bf16 = A8W8 block-scaled product of x[M,K] (bf16, quantised per token and
    128-block inside the call) and Wq[N,K] (e4m3 codes) with block scales sw."""
    M, K = x.shape
    N = Wq.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(DG_OP_GEMV_A8W8, M, N, K, device=x.device)
    _expect(x, "x", torch.bfloat16)
    _expect(Wq, "Wq", _FP8, (N, K))
    _expect(sw, "sw", torch.float32, ((N + 127) // 128, (K + 127) // 128))
    _expect(y, "y", torch.bfloat16, (M, N))
    _check_dev(x, Wq, sw, y, ws)
    _ok(lib().dg_gemv_a8w8_blockscale(_ptr(x), _ptr(Wq), _ptr(sw), _ptr(y), M, N, K, _ptr(ws), _nbytes(ws),
                                      _stream(stream), _choice(choice)), "dg_gemv_a8w8_blockscale")
    return y


def dg_quant_a8_blockscale(x, q=None, sx=None, stream=None):
    """(q [M,K] uint8 e4m3 codes, sx [M, ceil(K/128)] fp32): the A8W8 activation quantisation."""
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sx is None:
        sx = torch.empty((M, (K + 127) // 128), dtype=torch.float32, device=x.device)
    _expect(x, "x", torch.bfloat16)
    _expect(q, "q", _FP8, (M, K))
    _expect(sx, "sx", torch.float32, (M, (K + 127) // 128))
    _check_dev(x, q, sx)
    _ok(lib().dg_quant_a8_blockscale(_ptr(x), _ptr(q), _ptr(sx), M, K, _stream(stream)), "dg_quant_a8_blockscale")
    return q, sx


def dg_gate_up_silu(x, W_gu, out=None, ws=None, choice=None, stream=None):
    """out[M,N_half] = silu(x . W_gu[0::2]^T) * (x . W_gu[1::2]^T)."""
    M, K = x.shape
    Nh = W_gu.shape[0] // 2
    if out is None:
        out = torch.empty((M, Nh), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(DG_OP_GATE_UP_SILU, M, Nh, K, device=x.device)
    _expect(x, "x", torch.bfloat16)
    _expect(W_gu, "W_gu", torch.bfloat16, (2 * Nh, K))
    _expect(out, "out", torch.bfloat16, (M, Nh))
    _check_dev(x, W_gu, out, ws)
    _ok(lib().dg_gate_up_silu(_ptr(x), _ptr(W_gu), _ptr(out), M, Nh, K, _ptr(ws), _nbytes(ws),
                              _stream(stream), _choice(choice)), "dg_gate_up_silu")
    return out


def dg_head_fp8_argmax(x, Wq, scale, logits=None, argmax=None, ws=None, choice=None, stream=None,
                       want_logits=True):
    """(logits[M,N] bf16 or None, argmax[M] int32) for the fp8 head with one scale."""
    M, K = x.shape
    N = Wq.shape[0]
    if logits is None and want_logits:
        logits = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if argmax is None:
        argmax = torch.empty((M,), dtype=torch.int32, device=x.device)
    if ws is None:
        ws = workspace(DG_OP_HEAD_FP8_ARGMAX, M, N, K, device=x.device)
    _expect(x, "x", torch.bfloat16)
    _expect(Wq, "Wq", _FP8, (N, K))
    _expect(scale, "scale", torch.float32, min_numel=1)
    _expect(logits, "logits", torch.bfloat16, (M, N))
    _expect(argmax, "argmax", torch.int32, (M,))
    _check_dev(x, Wq, scale, logits, argmax, ws)
    _ok(lib().dg_head_fp8_argmax(_ptr(x), _ptr(Wq), _ptr(scale), _ptr(logits), _ptr(argmax), M, N, K,
                                 _ptr(ws), _nbytes(ws), _stream(stream), _choice(choice)),
        "dg_head_fp8_argmax")
    return logits, argmax


def dg_head_fp8_argmax_noalloc(x, Wq, scale, logits=None, argmax=None, choice=None, stream=None,
                               want_logits=True):
    """dg_head_fp8_argmax with the library's static scratch instead of a workspace."""
    M, K = x.shape
    N = Wq.shape[0]
    if logits is None and want_logits:
        logits = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if argmax is None:
        argmax = torch.empty((M,), dtype=torch.int32, device=x.device)
    _expect(x, "x", torch.bfloat16)
    _expect(Wq, "Wq", _FP8, (N, K))
    _expect(scale, "scale", torch.float32, min_numel=1)
    _expect(logits, "logits", torch.bfloat16, (M, N))
    _expect(argmax, "argmax", torch.int32, (M,))
    _check_dev(x, Wq, scale, logits, argmax)
    _ok(lib().dg_head_fp8_argmax_noalloc(_ptr(x), _ptr(Wq), _ptr(scale), _ptr(logits), _ptr(argmax), M, N,
                                         K, _stream(stream), _choice(choice)), "dg_head_fp8_argmax_noalloc")
    return logits, argmax


def dg_head_fp8_argmax_noalloc_status(stream=None) -> int:
    """The no-allocation head's status word (its latest call); synchronises the stream."""
    v = ctypes.c_int32(0)
    _ok(lib().dg_head_fp8_argmax_noalloc_status(ctypes.byref(v), _stream(stream)),
        "dg_head_fp8_argmax_noalloc_status")
    return int(v.value)


def dg_head_fp8_argmax_noalloc_scratch() -> int:
    """Device address of the no-allocation head's static scratch on the current device."""
    p = ctypes.c_void_p(0)
    _ok(lib().dg_head_fp8_argmax_noalloc_scratch(ctypes.byref(p)), "dg_head_fp8_argmax_noalloc_scratch")
    return int(p.value)


def dg_moe_w1_silu(x, topk_ids, W1, s1, a=None, ws=None, choice=None, stream=None):
    """a[M,topk,I] = silu(g) * u per routed slot."""
    M, K = x.shape
    topk = topk_ids.shape[1]
    E, twoI, _ = W1.shape
    I = twoI // 2
    if a is None:
        a = torch.empty((M, topk, I), dtype=torch.bfloat16, device=x.device)
    if ws is None:
        ws = workspace(DG_OP_MOE_W1, M, I, K, topk, device=x.device)
    _expect(x, "x", torch.bfloat16)
    _expect(topk_ids, "topk_ids", torch.int32, (M, topk))
    _expect(W1, "W1", _FP8, (E, 2 * I, K))
    _expect(s1, "s1", torch.float32, (E, 2 * I))
    _expect(a, "a", torch.bfloat16, (M, topk, I))
    _check_dev(x, topk_ids, W1, s1, a, ws)
    _ok(lib().dg_moe_w1_silu(_ptr(x), _ptr(topk_ids), _ptr(W1), _ptr(s1), _ptr(a), M, topk, E, I, K,
                             _ptr(ws), _nbytes(ws), _stream(stream), _choice(choice)), "dg_moe_w1_silu")
    return a


def dg_moe_w2(a, topk_ids, topk_w, W2, s2, y=None, ws=None, choice=None, stream=None):
    """y[M,Nout] = sum_k topk_w[t,k] * s2 * (a[t,k] . W2[e]^T)."""
    M, topk, I = a.shape
    E, Nout, _ = W2.shape
    if y is None:
        y = torch.empty((M, Nout), dtype=torch.bfloat16, device=a.device)
    if ws is None:
        ws = workspace(DG_OP_MOE_W2, M, Nout, I, topk, device=a.device)
    _expect(a, "a", torch.bfloat16)
    _expect(topk_ids, "topk_ids", torch.int32, (M, topk))
    _expect(topk_w, "topk_w", torch.float32, (M, topk))
    _expect(W2, "W2", _FP8, (E, Nout, I))
    _expect(s2, "s2", torch.float32, (E, Nout))
    _expect(y, "y", torch.bfloat16, (M, Nout))
    _check_dev(a, topk_ids, topk_w, W2, s2, y, ws)
    _ok(lib().dg_moe_w2(_ptr(a), _ptr(topk_ids), _ptr(topk_w), _ptr(W2), _ptr(s2), _ptr(y), M, topk, E,
                        I, Nout, _ptr(ws), _nbytes(ws), _stream(stream), _choice(choice)), "dg_moe_w2")
    return y


def dg_select(op: int, M: int, N: int, K: int) -> Choice:
    c = Choice()
    _ok(lib().dg_select(op, M, N, K, ctypes.byref(c)), "dg_select")
    return c


def dg_table_load(path: str):
    _ok(lib().dg_table_load(path.encode()), "dg_table_load")


def dg_table_clear():
    lib().dg_table_clear()


def dg_table_entries() -> int:
    return int(lib().dg_table_entries())


def dg_selection_space() -> int:
    return int(lib().dg_selection_space())


def dg_build_id() -> str:
    return lib().dg_build_id().decode()


def dg_table_check(path: str, arch: str, driver_version: int, runtime_version: int):
    """-> (status, entries, reason) without touching a GPU."""
    n = ctypes.c_int(0)
    buf = ctypes.create_string_buffer(512)
    s = lib().dg_table_check(path.encode(), arch.encode(), driver_version, runtime_version,
                             ctypes.byref(n), buf, 512)
    return int(s), int(n.value), buf.value.decode()


_OP_NAMES = ("gemv_bf16", "gate_up_silu", "head_fp8_argmax", "moe_w1_silu", "moe_w2", "gemv_a8w8")


def _bucket(M: int) -> int:
    for b in ROWS_BUCKETS:
        if b >= M:
            return b
    return -1


def _table_key(op_name: str, M: int, N: int, K: int):
    return (op_name, int(M), int(N), int(K))


def _sweep_remaining(shapes, doc):
    """The shapes whose (op, row bucket, N, K) entry a partial table does not hold yet."""
    have = {_table_key(e["op"], e["M"], e["N"], e["K"]) for e in doc.get("entries", [])}
    return [s for s in shapes if _table_key(_OP_NAMES[s[0]], _bucket(s[1]), s[2], s[3]) not in have]


def _merge_tables(old, new):
    """new's identity; old's entries that new does not re-measure, then new's."""
    fresh = {_table_key(e["op"], e["M"], e["N"], e["K"]) for e in new.get("entries", [])}
    kept = [e for e in old.get("entries", []) if _table_key(e["op"], e["M"], e["N"], e["K"]) not in fresh]
    out = dict(new)
    out["entries"] = kept + list(new.get("entries", []))
    return out


def _sweep_once(shapes, out_path, reps):
    arr = (Shape * len(shapes))(*[Shape(*s) for s in shapes])
    _ok(lib().dg_sweep(arr, len(shapes), out_path.encode(), reps), "dg_sweep")


def dg_sweep(shapes, out_path: str, reps: int = 20, resume: bool = False):
    """shapes: iterable of (op, M, N, K, topk[, E]); writes the shape table JSON to out_path.

    resume=True continues an interrupted sweep: when out_path already holds a table of
    this build and device (the same identity the new measurements get), its entries are
    kept and only the missing (op, row bucket, N, K) keys are measured; the merged table
    then replaces the file in one rename.  Any other file is measured over from scratch."""
    shapes = [tuple(s) for s in shapes]
    old = None
    if resume and os.path.exists(out_path):
        try:
            with open(out_path) as f:
                old = json.load(f)
        except (OSError, ValueError):
            old = None
        if not (isinstance(old, dict) and old.get("format") == "libdecodegemm-table"
                and old.get("identity", {}).get("build") == dg_build_id()
                and old.get("identity", {}).get("selection_space") == dg_selection_space()):
            old = None
    if old is None:
        _sweep_once(shapes, out_path, reps)
        return
    todo = _sweep_remaining(shapes, old)
    if not todo:
        return
    part = out_path + f".part{os.getpid()}"
    try:
        _sweep_once(todo, part, reps)
        with open(part) as f:
            new = json.load(f)
    finally:
        if os.path.exists(part):
            os.remove(part)
    if new.get("identity") != old.get("identity"):      # another device or driver: start over
        _sweep_once(shapes, out_path, reps)
        return
    tmp = out_path + f".tmp{os.getpid()}"
    with open(tmp, "w") as f:
        json.dump(_merge_tables(old, new), f, indent=1)
    os.replace(tmp, out_path)
