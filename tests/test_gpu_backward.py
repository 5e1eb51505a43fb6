"""GPU parity of the backward pass (dq, dk, dv, dMc through the C ABI)
against the float64 backward oracle.

Measure, per gradient: max|gpu - oracle| / max|oracle| over the whole
tensor.  Tolerances: dq, dk, dv are rounded to the tensors' dtype, so bf16
gets the forward's 5e-3.  dMc is a float32 sum over every head and token
whose terms cancel (sum_b Mc[i,b] dMc[i,b] = 0 under DIVISIVE; with one
block of 1000 tokens over 4 heads the terms are ~60 times the result).  The
tensor-core path (bf16 inputs) carries its float32 records as bf16 high +
low pairs (about 2^-17 relative) and drops the low x low product, so its
dMc gets 2e-3 (2^-16 times that cancellation, with margin); the float32
CUDA-core path gets 5e-4 with bf16 inputs and 5e-5 with float32 inputs.
Float32 dq, dk, dv get 2e-5: their DIVISIVE form is a difference of two
terms of the size of the output (dq = (S~ dO - z~ (dO . o)) / s).
"""

import zlib

import numpy as np
import pytest

from oracle import mhla_backward_oracle as orb
from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

from helpers import download, upload

pytestmark = pytest.mark.gpu

# dq, dk, dv take the forward's bounds (5e-3 bf16, 1e-5 float32; measured
# float32 worst 3.6e-6).  dMc[i, b] sums products over every unit and token of
# the blocks involved, and those terms cancel (under MALA the unit row sums,
# under DIVISIVE the invariance to scaling a row of Mc): its float32 error
# relative to its own largest entry reaches 2.0e-5 (MALA, two 1500-token
# blocks), hence 5e-5 there; bf16 inputs on the tensor cores keep hi + lo
# records (~2^-17 each) with the lo x lo product dropped, hence 2e-3.
TOL_X = {"bf16": 5e-3, "f32": 1e-5}
TOL_MC = {"bf16": 2e-3, "f32": 5e-5}
TOL_MC_SIMT_BF16 = 5e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from token_level_head_phi_gb300 import build
    build.build()
    mb.load()


def _gpu_backward(w, dev, gdev, mc, norm, fmap, variant="auto"):
    import torch
    q, k, v = upload(w, dev)
    (g,) = upload(w, [gdev])
    mct = torch.from_numpy(np.ascontiguousarray(mc, dtype=np.float32)).cuda()
    dq, dk, dv, dmc = mb.mhla_backward(q, k, v, mct, g, w.grid, w.block, norm=norm, feature_map=fmap,
                                     variant=variant)
    torch.cuda.synchronize()
    code, detail = mb.mhla_device_status()
    assert code == 0, f"device status {code} (detail {detail})"
    shape = (w.batch, w.heads, w.n_tokens, w.head_dim)
    return [download(x).reshape(shape) for x in (dq, dk, dv)] + [dmc.cpu().numpy().astype(np.float64)]


def backward_results(w, norm, fmap="elu1", mc=None, inputs=None, variant="auto"):
    """GPU and oracle gradients (dq, dk, dv, dMc) of the same seeded inputs,
    with the oracle's inputs and dO."""
    vals, dev = inputs if inputs is not None else wl.all_inputs(w)
    gvals, gdev = wl.output_grad(w)
    mc = wl.make_mc(w) if mc is None else mc
    got = _gpu_backward(w, dev, gdev, mc, norm, fmap, variant)
    want = orb.mhla_backward64(vals[0], vals[1], vals[2], np.asarray(mc, np.float64), w.grid, w.block, gvals,
                               fmap, norm)
    for name, x in zip(("dq", "dk", "dv", "dmc"), got):
        assert np.all(np.isfinite(x)), f"non-finite {name}"
    return got, want, vals, gvals, mc


def backward_parity(w, norm, fmap="elu1", mc=None, inputs=None, variant="auto"):
    """Worst relative error of (dq, dk, dv) and of dMc."""
    got, want, _, _, _ = backward_results(w, norm, fmap, mc, inputs, variant)
    ex = max(orc.relative_max_error(got[i], want[i]) for i in range(3))
    emc = orc.relative_max_error(got[3], want[3])
    return ex, emc


@pytest.mark.parametrize("variant", ["auto", "simt"])
@pytest.mark.parametrize("name,norm", [(n, m) for n in ("tiny_f32", "deit_t") for m in ("divisive", "none", "mala")]
                         + [("image_64x64", "divisive")])
def test_workload_backward(name, norm, variant):
    w = wl.WORKLOADS[name]
    if variant == "simt" and w.dtype == "f32":
        pytest.skip("float32 inputs always take the CUDA-core backward")
    ex, emc = backward_parity(w, norm, variant=variant)
    tol_mc = TOL_MC_SIMT_BF16 if (variant == "simt" and w.dtype == "bf16") else TOL_MC[w.dtype]
    assert ex <= TOL_X[w.dtype] and emc <= tol_mc, f"{name}/{norm}: {ex:.3e} {emc:.3e}"


@pytest.mark.parametrize("name", ["seq_32k_mala", "wan_21x30x50"])
def test_full_head_shape_backward(name):
    # the workloads' own grid, block and head shapes with two (batch, head) units
    w = wl.WORKLOADS[name].with_(batch=1, heads=2)
    ex, emc = backward_parity(w, w.norm)
    assert ex <= TOL_X[w.dtype] and emc <= TOL_MC[w.dtype], f"{name}: {ex:.3e} {emc:.3e}"


EDGE = [
    # grid, block, d, dtype, batch, heads
    ((1, 14, 14), (1, 7, 7), 64, "bf16", 1, 2),        # ragged 49-token blocks
    ((1, 10, 12), (1, 5, 4), 32, "f32", 2, 1),         # non-square blocks, d=32
    ((3, 8, 8), (3, 4, 8), 16, "f32", 1, 3),           # 3D, bt = T, d=16
    ((4, 6, 10), (2, 3, 5), 128, "bf16", 1, 1),        # 3D ragged, d=128
    ((2, 4, 8), (1, 2, 4), 128, "f32", 1, 2),          # d=128 in float32
    ((1, 1, 1000), (1, 1, 1000), 64, "bf16", 2, 2),    # one block (pieces of one block)
    ((1, 1, 3000), (1, 1, 1500), 64, "f32", 1, 1),     # two long blocks split into pieces
    ((1, 1, 4100), (1, 1, 41), 64, "bf16", 1, 1),      # M=100 odd blocks
    ((1, 9, 1), (1, 3, 1), 64, "bf16", 1, 1),          # column grid
    ((2, 2, 2), (1, 1, 1), 16, "f32", 1, 1),           # one token per block
    ((1, 1, 2304), (1, 1, 48), 64, "bf16", 1, 2),      # M=48: dMc tiles with a ragged edge
]


@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}-{c[3]}")
def test_edge_backward(case, norm):
    grid, block, d, dtype, batch, heads = case
    w = wl.random_small(zlib.crc32(repr(case).encode()) % 10000, grid, block, d, batch, heads, dtype)
    got, want, vals, gvals, mc = backward_results(w, norm)
    ex = max(orc.relative_max_error(got[i], want[i]) for i in range(3))
    if w.n_blocks == 1 and norm == "divisive":
        # One block: DIVISIVE is invariant to scaling a row of Mc, so o does
        # not depend on the single entry and dMc is zero up to rounding.  Its
        # two terms <dS~, S> and <dz~, z> are +T and -T per unit, T = sum_t
        # dO_t . o_t; the error is compared on the scale of those terms.
        scale = 0.0
        for u in range(w.units):
            b, h = divmod(u, w.heads)
            o = orc.mhla_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block)
            scale += float(np.abs(np.sum(gvals[b, h] * o, axis=1)).sum())
        emc = float(np.abs(got[3] - want[3]).max()) / scale
    else:
        emc = orc.relative_max_error(got[3], want[3])
    assert ex <= TOL_X[dtype] and emc <= TOL_MC[dtype], f"{case}/{norm}: {ex:.3e} {emc:.3e}"


def test_mc_with_zero_entries_backward():
    w = wl.random_small(5, (1, 16, 16), (1, 4, 4), 64, 2, 2, "bf16")
    M = w.n_blocks
    rng = np.random.default_rng(3)
    mc = rng.uniform(0, 1, (M, M)) * (rng.uniform(0, 1, (M, M)) < 0.3)
    np.fill_diagonal(mc, 1.0)
    mc = (mc / mc.sum(1, keepdims=True)).astype(np.float32)
    for norm in ("divisive", "mala", "none"):
        ex, emc = backward_parity(w, norm, mc=mc)
        assert ex <= TOL_X["bf16"] and emc <= TOL_MC["bf16"], f"{norm}: {ex:.3e} {emc:.3e}"


def test_identity_map_backward():
    w = wl.random_small(8, (1, 12, 12), (1, 4, 4), 64, 1, 2, "f32", mc="linear_decay")
    vals, _ = wl.all_inputs(w)
    vals = [np.abs(a) + 0.1 for a in vals]  # positive features for phi(x) = x
    dev = [a.astype(np.float32) for a in vals]
    for norm in ("divisive", "mala"):
        ex, emc = backward_parity(w, norm, fmap="identity", inputs=(vals, dev))
        assert ex <= TOL_X["f32"] and emc <= TOL_MC["f32"], f"{norm}: {ex:.3e} {emc:.3e}"


def test_backward_is_deterministic_and_leaves_guards():
    torch = pytest.importorskip("torch")
    w = wl.random_small(9, (1, 14, 14), (1, 7, 7), 64, 2, 3, "bf16")
    _, dev = wl.all_inputs(w)
    _, gdev = wl.output_grad(w)
    q, k, v = upload(w, dev)
    (g,) = upload(w, [gdev])
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    n = w.units * w.n_tokens * w.head_dim
    pad = 4096
    runs = []
    for _ in range(2):
        big = torch.full((3 * n + 2 * pad,), 777.0, dtype=torch.bfloat16, device="cuda")
        outs = [big[pad + i * n:pad + (i + 1) * n].view(q.shape) for i in range(3)]
        dmc = torch.empty_like(mc)
        mb.mhla_backward(q, k, v, mc, g, w.grid, w.block, dq=outs[0], dk=outs[1], dv=outs[2], dmc=dmc)
        torch.cuda.synchronize()
        assert torch.all(big[:pad] == 777.0) and torch.all(big[pad + 3 * n:] == 777.0)
        runs.append((big.clone(), dmc.clone()))
    assert torch.equal(runs[0][0].view(torch.int16), runs[1][0].view(torch.int16))
    assert torch.equal(runs[0][1], runs[1][1])


@pytest.mark.parametrize("variant", ["auto", "simt"])
@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("fmap", ["relu", "exp"])
def test_relu_and_exp_backward(fmap, norm, variant):
    w = wl.WORKLOADS["deit_t"].with_(batch=4)
    ex, emc = backward_parity(w, norm, fmap=fmap, variant=variant)
    tol_mc = TOL_MC_SIMT_BF16 if variant == "simt" else TOL_MC["bf16"]
    assert ex <= TOL_X["bf16"] and emc <= tol_mc, f"{fmap}/{norm}/{variant}: {ex:.3e} {emc:.3e}"


@pytest.mark.parametrize("variant", ["auto", "simt"])
@pytest.mark.parametrize("norm", ["divisive", "mala"])
def test_zero_denominator_rows_pass_no_gradient(norm, variant):
    w = wl.random_small(32, (1, 14, 14), (1, 7, 7), 64, 1, 2, "bf16")
    vals, _ = wl.all_inputs(w)
    q, k, v = (np.array(a) for a in vals)
    q[:, :, 3, :] = -np.abs(q[:, :, 3, :]) - 0.25   # phi(q_3) = 0 under ReLU
    pairs = [wl.round_to_bf16(a) for a in (q, k, v)]
    dev = [b for b, _ in pairs]
    vals = [x for _, x in pairs]
    ex, emc = backward_parity(w, norm, fmap="relu", inputs=(vals, dev), variant=variant)
    tol_mc = TOL_MC_SIMT_BF16 if variant == "simt" else TOL_MC["bf16"]
    assert ex <= TOL_X["bf16"] and emc <= tol_mc, f"{norm}/{variant}: {ex:.3e} {emc:.3e}"


@pytest.mark.parametrize("name", ["seq_32k", "wan_21x30x50"])
def test_full_size_backward_sampled_units(name):
    # the full workload in the launch configuration the bench times: dq, dk,
    # dv of sampled units against the oracle, and dMc through a property that
    # holds at any size -- under DIVISIVE the output is invariant to scaling a
    # row of Mc, so sum_b Mc[i,b] dMc[i,b] = 0 for every row i
    import torch
    w = wl.WORKLOADS[name]
    vals, dev = wl.all_inputs(w)
    gvals, gdev = wl.output_grad(w)
    mc = wl.make_mc(w)
    q, k, v = upload(w, dev)
    (g,) = upload(w, [gdev])
    dq, dk, dv, dmc = mb.mhla_backward(q, k, v, torch.from_numpy(mc).cuda(), g, w.grid, w.block, norm="divisive")
    torch.cuda.synchronize()
    code, detail = mb.mhla_device_status()
    assert code == 0, (code, detail)
    got = [download(x).reshape(w.units, w.n_tokens, w.head_dim) for x in (dq, dk, dv)]
    for u in (0, w.units - 1):
        b, h = divmod(u, w.heads)
        want = orb.mhla_head_backward64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block,
                                        gvals[b, h], "elu1", "divisive")
        for x, y in zip(got, want[:3]):
            assert orc.relative_max_error(x[u], y) <= TOL_X["bf16"], (name, u)
    dmc = dmc.cpu().numpy().astype(np.float64)
    terms = mc.astype(np.float64) * dmc
    assert np.all(np.isfinite(dmc))
    assert np.max(np.abs(terms.sum(axis=1))) <= 2e-3 * np.max(np.abs(terms).sum(axis=1))
