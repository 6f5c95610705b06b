"""Shared helpers for the CUDA-path tests."""
import re
import os

import numpy as np
import torch

from oracle import tolerance as T

# (max |gpu - ref| / bound, test) of every parity check in this session; the terminal
# summary lists the largest, so that drift towards the bound shows before it fails.
RATIOS = []


def _note(err, bound):
    err = np.asarray(err, np.float64)
    if err.size == 0:
        return
    r = float(np.max(err / np.asarray(bound, np.float64)))
    RATIOS.append((r, os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]))


def lin_excess(gpu, ref, absdot, rel=T.REL, abs_=T.ABS):
    """T.linear_excess, with the check's largest error/bound ratio recorded."""
    g = np.asarray(gpu, np.float64)
    _note(np.abs(g - ref), rel * np.asarray(absdot) + abs_)
    return T.linear_excess(g, ref, absdot, rel, abs_)


def silu_excess(gpu, g, u, absg, absu, ref):
    """T.silu_mul_excess, with the check's largest error/bound ratio recorded."""
    got = np.asarray(gpu, np.float64)
    _note(np.abs(got - ref), T.silu_mul_bound(g, u, absg, absu, ref))
    return T.silu_mul_excess(got, g, u, absg, absu, ref)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def sample_rows(N: int, n: int, seed: int) -> np.ndarray:
    """n distinct rows of [0, N), always including the first and last."""
    g = np.random.default_rng(seed)
    rows = set(g.choice(N, size=min(N, n), replace=False).tolist())
    rows.update({0, N - 1})
    return np.array(sorted(rows), dtype=np.int64)


def header_functions() -> list:
    """Every function name declared in include/*.h."""
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(inc, fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(dg_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))
