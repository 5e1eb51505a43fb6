"""GPU parity of the causal backward (dq, dk, dv, dMc of the block-ordered
causal form through the C ABI) against the float64 causal backward oracle.

Measure, per gradient: max|gpu - oracle| / max|oracle| over the whole
tensor.  The kernels are the float32 CUDA-core ones whatever the inputs'
dtype, so the bounds are those of the non-causal float32 backward: bf16
dq, dk, dv are rounded to bf16 (5e-3, the forward's bound), float32 ones
get 1e-5; dMc sums cancelling terms over every unit and token (5e-5 with
float32 inputs, 5e-4 with bf16 inputs, as for the non-causal CUDA-core
backward).  The diagonal of dMc is a sum over the block's tokens of
<dS~_t, R_t> + <dz~_t, rz_t> + <dv~_t, rv_t> + dn~_t rn_t, whose terms
cancel (with a single block DIVISIVE's output does not depend on Mc at all,
and they cancel exactly; a long MALA block cancels about a thousandfold):
float32 rounding there is relative to the sum of the terms' magnitudes, so
a diagonal entry may also stay within 64 float32 units of rounding (2^-24
each; dot products of up to 64 terms) of that sum.
"""

import zlib

import numpy as np
import pytest

from oracle import mhla_causal_backward_oracle as ocb
from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

from helpers import download, upload

pytestmark = pytest.mark.gpu

TOL_X = {"bf16": 5e-3, "f32": 1e-5}
TOL_MC = {"bf16": 5e-4, "f32": 5e-5}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from token_level_head_phi_gb300 import build
    build.build()
    mb.load()


def causal_backward_results(w, norm, fmap="elu1", mc=None, variant="auto", layout="bhnd"):
    import torch
    vals, dev = wl.all_inputs(w)
    gvals, gdev = wl.output_grad(w)
    mc = wl.make_mc(w) if mc is None else mc
    q, k, v = upload(w, dev)
    (g,) = upload(w, [gdev])
    shape = (w.batch, w.heads, w.n_tokens, w.head_dim)
    if layout == "bnhd":
        q, k, v, g = (x.permute(0, 2, 1, 3).contiguous() for x in (q, k, v, g))
    mct = torch.from_numpy(np.ascontiguousarray(mc, dtype=np.float32)).cuda()
    dq, dk, dv, dmc = mb.mhla_backward(q, k, v, mct, g, w.grid, w.block, norm=norm, feature_map=fmap,
                                       variant=variant, causal=True, layout=layout)
    torch.cuda.synchronize()
    code, detail = mb.mhla_device_status()
    assert code == 0, f"device status {code} (detail {detail})"
    if layout == "bnhd":
        dq, dk, dv = (x.permute(0, 2, 1, 3).contiguous() for x in (dq, dk, dv))
    got = [download(x).reshape(shape) for x in (dq, dk, dv)] + [dmc.cpu().numpy().astype(np.float64)]
    want = ocb.mhla_causal_backward64(vals[0], vals[1], vals[2], np.asarray(mc, np.float64), w.grid, w.block,
                                      gvals, fmap, norm)
    for name, x in zip(("dq", "dk", "dv", "dmc"), got):
        assert np.all(np.isfinite(x)), f"non-finite {name}"
    return got, want, vals, gvals, mc


def diag_term_magnitudes(w, vals, gvals, mc, fmap, norm):
    """Per head of Mc and block i: the sum over units and the block's tokens
    of |<dS~_t, R_t>| + |<dz~_t, rz_t>| + |<dv~_t, rv_t>| + |dn~_t rn_t|,
    the float64 terms whose sum is dMc[i, i]."""
    bidx = orc.block_of_token(w.grid, w.block)
    M = w.n_blocks
    mc = np.asarray(mc, np.float64)
    out = np.zeros((mc.shape[0], M) if mc.ndim == 3 else (1, M))
    for u in range(w.units):
        b, h = divmod(u, w.heads)
        mh, row = (mc[h], h) if mc.ndim == 3 else (mc, 0)
        phq = orc.feature_map(vals[0][b, h].astype(np.float64), fmap)
        phk = orc.feature_map(vals[1][b, h].astype(np.float64), fmap)
        vv = vals[2][b, h].astype(np.float64)
        g = gvals[b, h].astype(np.float64)
        S, z, vs, n = orc.block_summaries(phk, vv, bidx, M)
        Sp, zp, vp, npre = orc.mix(np.tril(mh, -1), S, z, vs, n)
        for i in range(M):
            wt = mh[i, i]
            R, rz, rv, rn = np.zeros_like(S[0]), np.zeros_like(z[0]), np.zeros_like(vs[0]), 0.0
            for t in np.nonzero(bidx == i)[0]:
                R += np.outer(phk[t], vv[t])
                rz += phk[t]
                rv += vv[t]
                rn += 1.0
                dnum, ds, dvt, dnt = ocb._token_grads(phq[t], g[t], Sp[i] + wt * R, zp[i] + wt * rz,
                                                      vp[i] + wt * rv, npre[i] + wt * rn, norm)
                out[row, i] += (abs(float(phq[t] @ R @ dnum)) + abs(ds * float(phq[t] @ rz))
                                + abs(float(np.dot(dvt, rv))) + abs(dnt * rn))
    return out


def errors(w, norm, got, want, vals, gvals, mc, fmap="elu1"):
    ex = max(orc.relative_max_error(got[i], want[i]) for i in range(3))
    top = float(np.abs(want[3]).max())
    mags = diag_term_magnitudes(w, vals, gvals, mc, fmap, norm)
    eye = np.eye(w.n_blocks, dtype=bool)
    diff = np.abs(got[3] - want[3]).reshape(-1, w.n_blocks, w.n_blocks)
    off = float(diff[:, ~eye].max()) / top if w.n_blocks > 1 else 0.0
    # a diagonal entry passes within TOL_MC * max|dMc| or 64 u * its magnitude sum
    cond = 64 * 2.0 ** -24 / TOL_MC[w.dtype]
    on = float((diff[:, eye] / np.maximum(cond * mags, top)).max())
    return ex, max(off, on)


@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("name", ["tiny_f32", "deit_t"])
def test_workload_causal_backward(name, norm):
    w = wl.WORKLOADS[name]
    got, want, vals, gvals, mc = causal_backward_results(w, norm)
    ex, emc = errors(w, norm, got, want, vals, gvals, mc)
    assert ex <= TOL_X[w.dtype] and emc <= TOL_MC[w.dtype], f"{name}/{norm}: {ex:.3e} {emc:.3e}"


EDGE = [
    # grid, block, d, dtype, batch, heads
    ((1, 14, 14), (1, 7, 7), 64, "bf16", 1, 2),        # ragged 49-token blocks (two tiles, a tail of 17)
    ((1, 10, 12), (1, 5, 4), 32, "f32", 2, 1),         # non-square blocks, d=32
    ((3, 8, 8), (3, 4, 8), 16, "f32", 1, 3),           # 3D, bt = T, d=16
    ((4, 6, 10), (2, 3, 5), 128, "bf16", 1, 1),        # 3D ragged, d=128 (16-token tiles)
    ((2, 4, 8), (1, 2, 4), 128, "f32", 1, 2),          # d=128 in float32
    ((1, 1, 1000), (1, 1, 1000), 64, "f32", 1, 2),     # one long block: the whole sequence in-block
    ((1, 1, 3000), (1, 1, 1500), 64, "f32", 1, 1),     # two long blocks kept as summary pieces
    ((1, 1, 4100), (1, 1, 41), 64, "bf16", 1, 1),      # M=100 odd blocks
    ((1, 9, 1), (1, 3, 1), 64, "bf16", 1, 1),          # column grid
    ((2, 2, 2), (1, 1, 1), 16, "f32", 1, 1),           # one token per block: no in-block pairs
    ((1, 1, 2304), (1, 1, 48), 64, "f32", 1, 2),       # M=48: dMc tiles with a ragged edge
]


@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}-{c[3]}")
def test_edge_causal_backward(case, norm):
    grid, block, d, dtype, batch, heads = case
    w = wl.random_small(zlib.crc32(repr(case).encode()) % 10000, grid, block, d, batch, heads, dtype)
    got, want, vals, gvals, mc = causal_backward_results(w, norm)
    ex, emc = errors(w, norm, got, want, vals, gvals, mc)
    assert ex <= TOL_X[dtype] and emc <= TOL_MC[dtype], f"{case}/{norm}: {ex:.3e} {emc:.3e}"
    # Mc above its diagonal does not enter the causal output
    assert np.all(np.triu(got[3], 1) == 0.0)


@pytest.mark.parametrize("norm", ["divisive", "mala"])
@pytest.mark.parametrize("fmap", ["relu", "exp"])
def test_relu_and_exp_causal_backward(fmap, norm):
    w = wl.random_small(31, (1, 8, 8), (1, 4, 4), 64, 2, 2, "f32")
    got, want, vals, gvals, mc = causal_backward_results(w, norm, fmap=fmap)
    ex, emc = errors(w, norm, got, want, vals, gvals, mc, fmap)
    assert ex <= TOL_X["f32"] and emc <= TOL_MC["f32"], f"{fmap}/{norm}: {ex:.3e} {emc:.3e}"


def test_token_major_and_per_head_mc_causal_backward():
    w = wl.random_small(12, (1, 8, 12), (1, 4, 4), 64, 2, 3, "f32")
    rng = np.random.default_rng(4)
    mc = rng.uniform(0.05, 1.0, (w.heads, w.n_blocks, w.n_blocks)).astype(np.float32)
    for layout in ("bhnd", "bnhd"):
        got, want, vals, gvals, _ = causal_backward_results(w, "mala", mc=mc, layout=layout)
        ex, emc = errors(w, "mala", got, want, vals, gvals, mc)
        assert got[3].shape == mc.shape
        assert ex <= TOL_X["f32"] and emc <= TOL_MC["f32"], f"{layout}: {ex:.3e} {emc:.3e}"


def test_causal_backward_only_reaches_earlier_tokens():
    # an upstream gradient on one token leaves every later token's dk, dv at 0
    import torch
    w = wl.random_small(17, (1, 6, 8), (1, 3, 4), 32, 1, 1, "f32")
    _, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mct = torch.from_numpy(wl.make_mc(w)).cuda()
    bidx = orc.block_of_token(w.grid, w.block)
    N = w.n_tokens
    order = np.argsort(bidx * N + np.arange(N), kind="stable")
    pos = np.empty(N, dtype=np.int64)
    pos[order] = np.arange(N)
    for t in (0, 13, 30):
        g = torch.zeros_like(q)
        g[0, 0, t] = 1.0
        dq, dk, dv, _ = mb.mhla_backward(q, k, v, mct, g, w.grid, w.block, norm="divisive", causal=True)
        torch.cuda.synchronize()
        later = torch.from_numpy(pos > pos[t]).cuda()
        assert torch.all(dk[0, 0][later] == 0) and torch.all(dv[0, 0][later] == 0)
        others = torch.ones(N, dtype=torch.bool, device="cuda")
        others[t] = False
        assert torch.all(dq[0, 0][others] == 0)


def test_causal_backward_rejects_tensor_core_variants():
    import torch
    w = wl.WORKLOADS["deit_t"]
    _, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mct = torch.from_numpy(wl.make_mc(w)).cuda()
    for variant in ("multipass", "fused"):
        with pytest.raises(RuntimeError, match="UNSUPPORTED|unsupported"):
            mb.mhla_backward(q, k, v, mct, q, w.grid, w.block, variant=variant, causal=True)
