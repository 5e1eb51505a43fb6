"""Seeded synthetic inputs for the MHLA forward pass.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic, so both the float64 oracle (through the tests) and
the CUDA path (through the tests and the benchmark) take their inputs from
here.  It imports numpy only.

Recipe (every config):
  * tokens live on a (T, Hg, Wg) grid in raster order, N = T*Hg*Wg;
  * for head unit u in [0, B*H) a generator ``default_rng([seed, 0, u])``
    draws Q_u, K_u, V_u in that order, each ``standard_normal((N, d))`` in
    float32, multiplied by the config's ``scale``;
  * bf16 configs round those float32 values to bf16 (round to nearest even)
    and both sides see the rounded values;
  * the block-mixing matrix Mc is drawn from ``default_rng([seed, 1])``.

The shapes follow the MHLA page (papernotes, "MHLA: Restoring Expressivity of
Linear Attention via Token-Level Multi-Head", experiments section): a
DeiT-T-like 14x14 patch grid with 3 heads of 64, DiT-like image token grids,
a Wan-like spatio-temporal grid and a 1D language-model sequence.  None of
those datasets or trained models is used: every value here is synthetic.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic MHLA problem: shapes, dtype, value scale, Mc recipe."""

    name: str
    batch: int
    heads: int
    head_dim: int
    grid: Tuple[int, int, int]   # (T, Hg, Wg); 1D sequences are (1, 1, N)
    block: Tuple[int, int, int]  # (bt, bh, bw)
    dtype: str                   # "bf16" or "f32"
    scale: float
    seed: int
    mc: str                      # "euclid_noise", "exp1d" or "linear_decay"
    norm: str = "divisive"       # default normalisation for this workload

    @property
    def n_tokens(self) -> int:
        return self.grid[0] * self.grid[1] * self.grid[2]

    @property
    def block_grid(self) -> Tuple[int, int, int]:
        return tuple(g // b for g, b in zip(self.grid, self.block))

    @property
    def n_blocks(self) -> int:
        bg = self.block_grid
        return bg[0] * bg[1] * bg[2]

    @property
    def block_tokens(self) -> int:
        return self.block[0] * self.block[1] * self.block[2]

    @property
    def units(self) -> int:
        """Independent (batch, head) problems."""
        return self.batch * self.heads

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five configurations of the benchmark (tiny fp32, DeiT-T-shaped,
# high-resolution image, video 3D grid, 1D long sequence).
WORKLOADS: Dict[str, Workload] = {
    "tiny_f32": Workload("tiny_f32", 1, 1, 16, (1, 8, 8), (1, 4, 4), "f32", 1.0, 1000, "euclid_noise"),
    "deit_t": Workload("deit_t", 64, 3, 64, (1, 14, 14), (1, 7, 7), "bf16", 1.0, 1001, "euclid_noise"),
    "image_64x64": Workload("image_64x64", 8, 8, 64, (1, 64, 64), (1, 8, 8), "bf16", 0.5, 1002, "euclid_noise"),
    "video_16x64x64": Workload("video_16x64x64", 2, 16, 64, (16, 64, 64), (2, 8, 8), "bf16", 1.0, 1003, "euclid_noise"),
    "seq_32k": Workload("seq_32k", 4, 16, 64, (1, 1, 32768), (1, 1, 256), "bf16", 1.0, 1004, "exp1d"),
    "seq_32k_mala": Workload("seq_32k_mala", 4, 16, 64, (1, 1, 32768), (1, 1, 256), "bf16", 1.0, 1004, "exp1d", "mala"),
    "seq_32k_m1": Workload("seq_32k_m1", 4, 16, 64, (1, 1, 32768), (1, 1, 32768), "bf16", 1.0, 1004, "exp1d"),
    "seq_32k_m1_mala": Workload("seq_32k_m1_mala", 4, 16, 64, (1, 1, 32768), (1, 1, 32768), "bf16", 1.0, 1004, "exp1d", "mala"),
    # video sequence of the length and block count the MHLA page reports for
    # Wan (31.5k tokens, M = 105): 21 x 30 x 50 grid, 3 x 10 x 10 blocks of 300
    # tokens (not a multiple of the 128-row tile: three 100-token chunks each)
    "wan_21x30x50": Workload("wan_21x30x50", 2, 12, 64, (21, 30, 50), (3, 10, 10), "bf16", 1.0, 1005, "euclid_noise"),
}

BENCH_WORKLOAD = "video_16x64x64"


def round_to_bf16(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Round float32 values to bf16 (nearest, ties to even).

    Returns ``(bits, values)``: the uint16 bit patterns to upload and the
    same numbers as float32, which is what the oracle reads.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    vals = r.view(np.float32)
    bits = (r >> np.uint32(16)).astype(np.uint16)
    return bits, vals


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _block_centres(w: Workload) -> np.ndarray:
    """Centre of every block in block-index units, blocks in raster order."""
    gt, gh, gw = w.block_grid
    t, y, x = np.meshgrid(np.arange(gt), np.arange(gh), np.arange(gw), indexing="ij")
    return np.stack([t.ravel(), y.ravel(), x.ravel()], axis=1).astype(np.float64)


def make_mc(w: Workload, kind: Optional[str] = None) -> np.ndarray:
    """Block-mixing coefficients Mc [M, M] (float32, rows sum to 1).

    Row i belongs to query block i, column b to summary block b.
      euclid_noise : exp(-||c_i - c_b|| / 2) + U(0, 0.05), then rows normalised
      exp1d        : exp(-|i - b| / 4), rows normalised (1D sequences)
      linear_decay : the locality-biased initialisation of the MHLA page
                     (key design 3): 1 - dist(i,b) / max_k dist(i,k), rows
                     normalised; with a single block Mc = [[1]].
    """
    kind = kind or w.mc
    M = w.n_blocks
    c = _block_centres(w)
    dist = np.sqrt(((c[:, None, :] - c[None, :, :]) ** 2).sum(-1))
    if kind == "euclid_noise":
        rng = np.random.default_rng([w.seed, 1])
        m = np.exp(-dist / 2.0) + rng.uniform(0.0, 0.05, size=(M, M))
    elif kind == "exp1d":
        i = np.arange(M, dtype=np.float64)
        m = np.exp(-np.abs(i[:, None] - i[None, :]) / 4.0)
    elif kind == "linear_decay":
        if M == 1:
            m = np.ones((1, 1))
        else:
            m = 1.0 - dist / dist.max(axis=1, keepdims=True)
    else:
        raise ValueError(f"unknown Mc recipe {kind!r}")
    m = m / m.sum(axis=1, keepdims=True)
    return m.astype(np.float32)


def head_qkv(w: Workload, unit: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Float32 Q, K, V [N, d] of one (batch, head) unit, before any rounding."""
    rng = np.random.default_rng([w.seed, 0, unit])
    shape = (w.n_tokens, w.head_dim)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    if w.scale != 1.0:
        s = np.float32(w.scale)
        q *= s
        k *= s
        v *= s
    return q, k, v


def head_inputs(w: Workload, unit: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Q, K, V [N, d] of one unit as the device sees them (bf16-rounded if bf16)."""
    q, k, v = head_qkv(w, unit)
    if w.dtype == "bf16":
        q, k, v = (round_to_bf16(a)[1] for a in (q, k, v))
    return q, k, v


def all_inputs(w: Workload):
    """Every unit's inputs, [B, H, N, d].

    Returns ``(arrays, device_arrays)``: float32 values (what the oracle
    reads) and the arrays to upload (uint16 bf16 bits, or float32).
    """
    U, N, d = w.units, w.n_tokens, w.head_dim
    vals = [np.empty((U, N, d), np.float32) for _ in range(3)]
    dev = [np.empty((U, N, d), np.uint16 if w.dtype == "bf16" else np.float32) for _ in range(3)]
    for u in range(U):
        for a, (x, dv) in enumerate(zip(head_qkv(w, u), dev)):
            if w.dtype == "bf16":
                bits, rounded = round_to_bf16(x)
                dv[u] = bits
                vals[a][u] = rounded
            else:
                dv[u] = x
                vals[a][u] = x
    shape = (w.batch, w.heads, N, d)
    return [x.reshape(shape) for x in vals], [x.reshape(shape) for x in dev]


def all_device_inputs(w: Workload):
    """Only the arrays to upload, [B, H, N, d] (saves the float32 copies)."""
    U, N, d = w.units, w.n_tokens, w.head_dim
    dt = np.uint16 if w.dtype == "bf16" else np.float32
    dev = [np.empty((U, N, d), dt) for _ in range(3)]
    for u in range(U):
        for x, dv in zip(head_qkv(w, u), dev):
            dv[u] = round_to_bf16(x)[0] if w.dtype == "bf16" else x
    shape = (w.batch, w.heads, N, d)
    return [x.reshape(shape) for x in dev]


def output_grad(w: Workload):
    """Seeded upstream gradient dO [B, H, N, d] for the backward pass (standard
    normal values, rounded to bf16 for bf16 workloads).

    Returns ``(values, device_array)`` like ``all_inputs``.
    """
    U, N, d = w.units, w.n_tokens, w.head_dim
    vals = np.empty((U, N, d), np.float32)
    dev = np.empty((U, N, d), np.uint16 if w.dtype == "bf16" else np.float32)
    for u in range(U):
        x = np.random.default_rng([w.seed, 1, u]).standard_normal((N, d), dtype=np.float32)
        if w.dtype == "bf16":
            dev[u], vals[u] = round_to_bf16(x)
        else:
            dev[u] = vals[u] = x
    shape = (w.batch, w.heads, N, d)
    return vals.reshape(shape), dev.reshape(shape)


def head_output_grad(w: Workload, unit: int) -> np.ndarray:
    """dO [N, d] of one unit as the device sees it (the values of output_grad)."""
    x = np.random.default_rng([w.seed, 1, unit]).standard_normal((w.n_tokens, w.head_dim), dtype=np.float32)
    return round_to_bf16(x)[1] if w.dtype == "bf16" else x


def random_small(seed: int, grid, block, d: int, batch: int = 1, heads: int = 1,
                 dtype: str = "f32", scale: float = 1.0, mc: str = "euclid_noise") -> Workload:
    """A small ad-hoc workload for edge-case tests."""
    return Workload(f"small_{seed}", batch, heads, d, tuple(grid), tuple(block), dtype, scale, seed, mc)


def roofline_bytes(w: Workload) -> int:
    """Bytes the method has to move: read Q, K, V, write O, read Mc once."""
    el = 2 if w.dtype == "bf16" else 4
    return 4 * w.units * w.n_tokens * w.head_dim * el + 4 * w.n_blocks ** 2


def roofline_flops(w: Workload) -> int:
    """Dense FLOPs: 4*N*d^2 (summaries + output) + 2*M^2*d^2 (mixing) per unit."""
    N, d, M = w.n_tokens, w.head_dim, w.n_blocks
    return w.units * (4 * N * d * d + 2 * M * M * d * d)


def backward_roofline_bytes(w: Workload) -> int:
    """Bytes the backward has to move: read Q, K, V, dO and Mc, write dQ, dK,
    dV and dMc."""
    el = 2 if w.dtype == "bf16" else 4
    return 7 * w.units * w.n_tokens * w.head_dim * el + 8 * w.n_blocks ** 2


def backward_roofline_flops(w: Workload) -> int:
    """Dense FLOPs of the backward per unit: the forward summaries and mixing
    recomputed (2*N*d^2 + 2*M^2*d^2), the output step (phi(q) S~, dq and dS~:
    6*N*d^2), the gradient mixing and dMc (4*M^2*d^2) and dk, dv (4*N*d^2)."""
    N, d, M = w.n_tokens, w.head_dim, w.n_blocks
    return w.units * (12 * N * d * d + 6 * M * M * d * d)


def describe(w: Workload) -> dict:
    return {
        "workload": w.name, "batch": w.batch, "heads": w.heads, "head_dim": w.head_dim,
        "grid": list(w.grid), "block": list(w.block), "n_tokens": w.n_tokens,
        "n_blocks": w.n_blocks, "dtype": w.dtype, "norm": w.norm, "mc": w.mc,
        "seed": w.seed, "scale": w.scale,
    }


__all__ = [
    "Workload", "WORKLOADS", "BENCH_WORKLOAD", "round_to_bf16", "bf16_bits_to_f32",
    "make_mc", "head_qkv", "head_inputs", "all_inputs", "all_device_inputs",
    "random_small", "roofline_bytes", "roofline_flops", "describe",
]
