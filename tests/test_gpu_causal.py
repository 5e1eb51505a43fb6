"""GPU parity of the block-ordered causal form against the causal float64
oracle, on the tensor-core path (bf16, d = 64, DIVISIVE / NONE: AUTO) and
the float32 CUDA-core kernels (SIMT); same measure and tolerances as the
non-causal parity tests (max|gpu - oracle| / max|oracle| per unit)."""

import zlib

import numpy as np
import pytest

from oracle import mhla_causal_oracle as occ
from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

from helpers import TOL, download, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from token_level_head_phi_gb300 import build
    build.build()
    mb.load()


def causal_parity(w, norm, fmap="elu1", units=None, mc=None, variant="auto"):
    import torch
    vals, dev = wl.all_inputs(w)
    mc = wl.make_mc(w) if mc is None else mc
    q, k, v = upload(w, dev)
    mct = torch.from_numpy(np.ascontiguousarray(mc, dtype=np.float32)).cuda()
    o = mb.mhla_forward(q, k, v, mct, w.grid, w.block, norm=norm, feature_map=fmap, causal=True, variant=variant)
    torch.cuda.synchronize()
    code, detail = mb.mhla_device_status()
    assert code == 0, f"device status {code} (detail {detail})"
    o = download(o).reshape(w.units, w.n_tokens, w.head_dim)
    worst = 0.0
    for u in (range(w.units) if units is None else units):
        b, h = divmod(u, w.heads)
        want = occ.mhla_causal_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block, fmap, norm)
        assert np.all(np.isfinite(o[u]))
        worst = max(worst, orc.relative_max_error(o[u], want))
    return worst


@pytest.mark.parametrize("variant", ["auto", "simt"])
@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("name", ["tiny_f32", "deit_t"])
def test_workload_causal(name, norm, variant):
    w = wl.WORKLOADS[name]
    err = causal_parity(w, norm, units=[0, w.units - 1], variant=variant)
    assert err <= TOL[w.dtype], f"{name}/{norm}: {err:.3e}"


@pytest.mark.parametrize("variant", ["auto", "simt"])
@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
def test_sequence_head_causal(norm, variant):
    # the 1D language-model shape: 128 blocks of 256 tokens (two 128-token
    # chunks per block on the tensor cores, eight 32-token tiles in float32)
    w = wl.WORKLOADS["seq_32k"].with_(batch=1, heads=2)
    err = causal_parity(w, norm, variant=variant)
    assert err <= TOL[w.dtype], f"{norm}: {err:.3e}"


EDGE = [
    # grid, block, d, dtype, batch, heads
    ((1, 14, 14), (1, 7, 7), 64, "bf16", 1, 2),        # 49-token blocks: ragged last tile
    ((4, 16, 16), (2, 8, 8), 64, "bf16", 1, 2),        # video-shaped 128-token blocks (one chunk)
    ((1, 1, 2100), (1, 1, 300), 64, "bf16", 1, 2),     # 300-token 1D blocks: three 100-token chunks
    ((3, 10, 10), (3, 10, 10), 64, "bf16", 1, 1),      # one 300-token 3D block: chunks of whole planes
    ((1, 1, 1000), (1, 1, 1000), 64, "bf16", 1, 1),    # one long block: eight chunks
    ((1, 1, 300), (1, 1, 100), 32, "f32", 1, 2),       # 1D, 100-token blocks
    ((3, 8, 8), (3, 4, 8), 16, "f32", 1, 1),           # 3D blocks
    ((2, 4, 8), (1, 2, 4), 128, "bf16", 1, 1),         # d = 128
    ((1, 1, 64), (1, 1, 64), 64, "f32", 2, 1),         # one block: textbook causal linear attention
    ((2, 2, 2), (1, 1, 1), 16, "f32", 1, 1),           # one token per block: pure block causality
]


@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}-{c[3]}")
def test_edge_causal(case, norm):
    grid, block, d, dtype, batch, heads = case
    w = wl.random_small(zlib.crc32(repr(case).encode()) % 10000, grid, block, d, batch, heads, dtype)
    err = causal_parity(w, norm)
    assert err <= TOL[dtype], f"{case}/{norm}: {err:.3e}"


@pytest.mark.parametrize("fmap", ["relu", "exp"])
def test_causal_feature_maps(fmap):
    w = wl.random_small(41, (1, 1, 512), (1, 1, 64), 64, 1, 2, "bf16")
    for norm in ("divisive", "mala"):
        err = causal_parity(w, norm, fmap=fmap)
        assert err <= TOL["bf16"], f"{fmap}/{norm}: {err:.3e}"


def test_causal_outputs_ignore_later_tokens():
    # changing K, V of the second half of a 1D sequence leaves the first half's
    # outputs bit-identical
    import torch
    w = wl.random_small(42, (1, 1, 1024), (1, 1, 128), 64, 1, 2, "bf16")
    _, dev = wl.all_inputs(w)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    q, k, v = upload(w, dev)
    a = mb.mhla_forward(q, k, v, mc, w.grid, w.block, causal=True).clone()
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 512:] = 1.5
    v2[:, :, 512:] = -3.0
    b = mb.mhla_forward(q, k2, v2, mc, w.grid, w.block, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[:, :, :512].view(torch.int16), b[:, :, :512].view(torch.int16))
    assert not torch.equal(a[:, :, 512:].view(torch.int16), b[:, :, 512:].view(torch.int16))
