"""Shared helpers for the CUDA-path tests."""
import re
import os

import numpy as np
import torch

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
