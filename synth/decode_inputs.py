"""Seeded synthetic workloads for the decode-time skinny linears.

Every generator takes an explicit seed (derived from the op and shape by
``seed_for``) and a device; the same call gives the same bytes on CPU each time,
so the CUDA path and the oracle are fed identical inputs.

Recipes (the distributions the workloads are specified with):
  * bf16 linear: x ~ N(0,1) [M,K], W ~ N(0,1/K) [N,K] row-major, both rounded to bf16.
  * fused gate/up: W_gate, W_up ~ N(0,1/K) [N_half,K], stored row-interleaved as one
    [2*N_half, K] matrix: row 2j is gate row j, row 2j+1 is up row j.
  * fp8 head: W ~ N(0,1/K) [N,K] quantised to e4m3 (OCP "fn" variant) with one fp32
    scale = max|W|/448; x ~ N(0,1) bf16 [M,K].
  * MoE: per token, ``topk`` distinct experts drawn uniformly without replacement,
    ``topk`` scores ~ N(0,1) turned into gate weights by a softmax (fp64, stored fp32);
    W1 [E, 2I, K] and W2 [E, Nout, I] ~ N(0, 1/K_in) quantised to e4m3 with one fp32
    scale per output row (max over that row / 448).
  * A8W8 blockscale linear: x ~ N(0,1) bf16 [M,K]; W ~ N(0,1/K) [N,K] quantised to e4m3
    with one fp32 scale per 128 x 128 block (max over the block / 448).

Quantisation here is input preparation (it produces the bytes the kernels read);
it uses torch's own float8_e4m3fn cast after clamping to the finite range.
"""
from __future__ import annotations

import zlib

import torch

E4M3_MAX = 448.0

__all__ = [
    "seed_for", "normal_bf16", "linear_inputs", "gate_up_inputs", "quantize_e4m3_per_tensor",
    "quantize_e4m3_per_row", "head_inputs", "moe_routing", "moe_weights", "moe_inputs", "E4M3_MAX",
    "quantize_e4m3_blocks", "a8w8_inputs",
]


def seed_for(*parts) -> int:
    """Stable 31-bit seed from any printable parts (op name, shape, M, ...)."""
    return zlib.crc32("|".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def linear_inputs(M: int, N: int, K: int, device="cpu", tag: str = "gemv_bf16"):
    """x [M,K] ~ N(0,1), W [N,K] ~ N(0,1/K), both bf16."""
    W = normal_bf16((N, K), K ** -0.5, seed_for(tag, "W", N, K), device)
    x = normal_bf16((M, K), 1.0, seed_for(tag, "x", N, K, M), device)
    return x, W


def gate_up_inputs(M: int, N_half: int, K: int, device="cpu"):
    """x [M,K]; W_gu [2*N_half, K] with gate row j at 2j and up row j at 2j+1."""
    Wg = normal_bf16((N_half, K), K ** -0.5, seed_for("gate", N_half, K), device)
    Wu = normal_bf16((N_half, K), K ** -0.5, seed_for("up", N_half, K), device)
    W = torch.stack((Wg, Wu), dim=1).reshape(2 * N_half, K).contiguous()
    x = normal_bf16((M, K), 1.0, seed_for("gate_up_x", N_half, K, M), device)
    return x, W


def _to_e4m3_bytes(v: torch.Tensor) -> torch.Tensor:
    return v.clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def quantize_e4m3_per_tensor(w: torch.Tensor):
    """fp32 tensor -> (uint8 e4m3 codes, fp32 scale tensor of shape [1]); scale = max|w|/448."""
    amax = w.abs().max().to(torch.float32)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).reshape(1)
    q = _to_e4m3_bytes(w / scale)
    return q, scale


def quantize_e4m3_per_row(w: torch.Tensor):
    """fp32 tensor [..., n, k] -> (uint8 codes, fp32 scales [..., n]); one scale per row."""
    amax = w.abs().amax(dim=-1).to(torch.float32)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = _to_e4m3_bytes(w / scale.unsqueeze(-1))
    return q, scale


def head_inputs(M: int, N: int, K: int, device="cpu", chunk_rows: int = 16384):
    """x [M,K] bf16; Wq [N,K] uint8 e4m3 codes; scale fp32 [1] (per tensor)."""
    seedW = seed_for("head", "W", N, K)
    # Draw W in row chunks (bounded peak memory), two passes: max first, then quantise.
    std = K ** -0.5
    amax = torch.zeros((), dtype=torch.float32, device=device)
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        w = torch.randn((r1 - r0, K), generator=_gen(seedW + r0, device), device=device) * std
        amax = torch.maximum(amax, w.abs().max())
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).reshape(1)
    Wq = torch.empty((N, K), dtype=torch.uint8, device=device)
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        w = torch.randn((r1 - r0, K), generator=_gen(seedW + r0, device), device=device) * std
        Wq[r0:r1] = _to_e4m3_bytes(w / scale)
    x = normal_bf16((M, K), 1.0, seed_for("head", "x", N, K, M), device)
    return x, Wq, scale


def moe_routing(M: int, topk: int, E: int, seed: int):
    """topk_ids [M,topk] int32 (distinct per token), topk_w [M,topk] fp32 (softmax of N(0,1))."""
    g = _gen(seed, "cpu")
    ids = torch.empty((M, topk), dtype=torch.int32)
    for t in range(M):
        ids[t] = torch.randperm(E, generator=g)[:topk].to(torch.int32)
    scores = torch.randn((M, topk), generator=g, dtype=torch.float64)
    w = torch.softmax(scores, dim=-1).to(torch.float32)
    return ids, w


def moe_weights(E: int, I: int, K: int, Nout: int, device="cpu"):
    """W1 [E,2I,K] (gate rows 0..I-1, up rows I..2I-1), s1 [E,2I]; W2 [E,Nout,I], s2 [E,Nout]."""
    W1q = torch.empty((E, 2 * I, K), dtype=torch.uint8, device=device)
    s1 = torch.empty((E, 2 * I), dtype=torch.float32, device=device)
    W2q = torch.empty((E, Nout, I), dtype=torch.uint8, device=device)
    s2 = torch.empty((E, Nout), dtype=torch.float32, device=device)
    for e in range(E):
        w1 = torch.randn((2 * I, K), generator=_gen(seed_for("moe_W1", e, I, K), device),
                         device=device) * K ** -0.5
        W1q[e], s1[e] = quantize_e4m3_per_row(w1)
        w2 = torch.randn((Nout, I), generator=_gen(seed_for("moe_W2", e, Nout, I), device),
                         device=device) * I ** -0.5
        W2q[e], s2[e] = quantize_e4m3_per_row(w2)
    return W1q, s1, W2q, s2


def moe_inputs(M: int, K: int, topk: int, E: int, rep: int = 0, device="cpu"):
    """x [M,K] bf16, topk_ids [M,topk] int32, topk_w [M,topk] fp32 (routing on CPU, then moved)."""
    x = normal_bf16((M, K), 1.0, seed_for("moe_x", M, K, rep), device)
    ids, w = moe_routing(M, topk, E, seed_for("moe_route", M, topk, E, rep))
    return x, ids.to(device), w.to(device)


def quantize_e4m3_blocks(w: torch.Tensor, block: int = 128):
    """fp32 [N, K] -> (uint8 e4m3 codes [N, K], fp32 scales [ceil(N/128), ceil(K/128)]);
    one scale per 128 x 128 block, max|w|/448 of the block (1 for an all-zero block)."""
    N, K = w.shape
    nbn, nbk = (N + block - 1) // block, (K + block - 1) // block
    pad = torch.zeros((nbn * block, nbk * block), dtype=torch.float32, device=w.device)
    pad[:N, :K] = w
    blocks = pad.view(nbn, block, nbk, block)
    amax = blocks.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = _to_e4m3_bytes(blocks / scale[:, None, :, None]).view(nbn * block, nbk * block)[:N, :K].contiguous()
    return q, scale.contiguous()


def a8w8_inputs(M: int, N: int, K: int, device="cpu", chunk_rows: int = 8192):
    """x [M,K] bf16 ~ N(0,1); Wq [N,K] e4m3 codes and sw [ceil(N/128), ceil(K/128)] fp32 from
    W ~ N(0, 1/K) quantised per 128 x 128 block (row chunks of 128 rows keep memory bounded)."""
    seedW = seed_for("a8w8", "W", N, K)
    Wq = torch.empty((N, K), dtype=torch.uint8, device=device)
    sw = torch.empty(((N + 127) // 128, (K + 127) // 128), dtype=torch.float32, device=device)
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        w = torch.randn((r1 - r0, K), generator=_gen(seedW + r0, device), device=device) * K ** -0.5
        q, s = quantize_e4m3_blocks(w)
        Wq[r0:r1] = q
        sw[r0 // 128:(r1 + 127) // 128] = s
    x = normal_bf16((M, K), 1.0, seed_for("a8w8", "x", N, K, M), device)
    return x, Wq, sw
