"""GPU parity of the tensor-core path at input scales far from unit size.

The block summaries S_b and z_b are plain sums with no range restriction
("MHLA: Restoring Expressivity of Linear Attention via Token-Level
Multi-Head", overall framework), so the output must follow the oracle for
any finite inputs: tiny and large values, steep ELU+1 features, exponential
features of large keys, a single dominant token, and Mc rows with zeros.
DIVISIVE is invariant to the scale of V's unit, NONE and MALA scale with it;
every case compares against the float64 oracle with the bf16 bound
(max|gpu - oracle| / max|oracle| <= 5e-3) and checks that the device status
stays clean (no call reports an error on inputs whose oracle output is
finite).
"""

import numpy as np
import pytest

from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

from helpers import TOL, download, run_gpu, upload

pytestmark = pytest.mark.gpu

NORMS = ["divisive", "none", "mala"]
VARIANTS = ["multipass", "fused"]
SHAPES = {
    # grid, block, batch, heads: 2D blocks of 32 tokens, 1D blocks of two
    # 128-token chunks, 3D video-like blocks of 128
    "2d": ((1, 16, 16), (1, 4, 8), 2, 3),
    "1d": ((1, 1, 2048), (1, 1, 256), 1, 2),
    "3d": ((4, 16, 16), (2, 8, 8), 1, 2),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from token_level_head_phi_gb300 import build
    build.build()
    mb.load()


def rescaled(w, sq=1.0, sk=1.0, sv=1.0, kmax=None, edit=None):
    """The workload's seeded inputs with Q, K, V multiplied by sq, sk, sv (K
    rescaled so that max|K| = kmax when given; `edit(q, k, v)` may change
    them in place), rounded to bf16.  Returns (oracle values, device bits)."""
    vals, _ = wl.all_inputs(w)
    q, k, v = (np.array(a, dtype=np.float64) for a in vals)
    q *= sq
    k *= sk
    v *= sv
    if kmax is not None:
        k *= kmax / np.abs(k).max()
    if edit is not None:
        edit(q, k, v)
    pairs = [wl.round_to_bf16(a.astype(np.float32)) for a in (q, k, v)]
    return [x for _, x in pairs], [b for b, _ in pairs]


def check(w, vals, dev, norm, variant, fmap="elu1", mc=None, units=None):
    mc = wl.make_mc(w) if mc is None else mc
    o = download(run_gpu(w, upload(w, dev), mc, norm, variant, fmap)).reshape(w.units, w.n_tokens, w.head_dim)
    worst = 0.0
    for u in (range(w.units) if units is None else units):
        b, h = divmod(u, w.heads)
        want = orc.mhla_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block, fmap, norm)
        assert np.all(np.isfinite(want)), "the oracle output must be finite for these inputs"
        assert np.all(np.isfinite(o[u])), f"non-finite output in unit {u}"
        worst = max(worst, orc.relative_max_error(o[u], want))
    return worst


def small(shape, seed):
    grid, block, batch, heads = SHAPES[shape]
    return wl.random_small(seed, grid, block, 64, batch, heads, "bf16")


CASES = {
    # name: (feature map, rescaled() keywords)
    "v_1e-6": ("elu1", dict(sv=1e-6)),
    "v_1e3": ("elu1", dict(sv=1e3)),
    "v_1e-30": ("elu1", dict(sv=1e-30)),
    "k_x8": ("elu1", dict(sk=8.0)),
    "q_x8_k_x8": ("elu1", dict(sq=8.0, sk=8.0)),
    "exp_k_to_20": ("exp", dict(kmax=20.0)),
    "exp_k_to_20_v_1e-4": ("exp", dict(kmax=20.0, sv=1e-4)),
}


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("shape", list(SHAPES))
def test_scaled_inputs(shape, case, norm, variant):
    fmap, kw = CASES[case]
    w = small(shape, 400 + len(case))
    vals, dev = rescaled(w, **kw)
    err = check(w, vals, dev, norm, variant, fmap)
    assert err <= TOL["bf16"], f"{shape}/{case}/{norm}/{variant}: rel err {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("norm", NORMS)
def test_one_dominant_token_and_zero_weights(norm, variant):
    """Exponential features with one key at +20 in the first block (its block
    summary is ~e^20 times the others) and the locality-decay Mc, whose rows
    give the farthest blocks weight exactly 0: rows that never see the
    dominant block keep their own precision."""
    w = wl.random_small(41, (1, 16, 16), (1, 4, 4), 64, 1, 2, "bf16", mc="linear_decay")

    def edit(q, k, v):
        k[:, :, 0, :] = 20.0

    vals, dev = rescaled(w, edit=edit)
    mc = wl.make_mc(w)
    assert (mc == 0).any(), "the decay Mc gives the farthest blocks weight 0"
    err = check(w, vals, dev, norm, variant, "exp", mc=mc)
    assert err <= TOL["bf16"], f"{norm}/{variant}: rel err {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("norm", NORMS)
def test_blocks_of_very_different_scales(norm, variant):
    """Each block's V carries its own scale, 10^-8 .. 10^3 across the blocks,
    so the records of one head span eleven decades.  With Mc = I every query
    block sees only its own block, and each block's output is compared on its
    own scale: no block's summary may lose precision to another's."""
    w = wl.random_small(43, (1, 16, 16), (1, 4, 8), 64, 1, 2, "bf16")
    scales = 10.0 ** np.linspace(-8, 3, w.n_blocks)
    blk = np.array([(t // 16 // 4) * 2 + (t % 16) // 8 for t in range(w.n_tokens)])

    def edit(q, k, v):
        v *= scales[blk][None, None, :, None]

    vals, dev = rescaled(w, edit=edit)
    mc = np.eye(w.n_blocks, dtype=np.float32)
    o = download(run_gpu(w, upload(w, dev), mc, norm, variant)).reshape(w.units, w.n_tokens, w.head_dim)
    for u in range(w.units):
        want = orc.mhla_head64(vals[0][0, u], vals[1][0, u], vals[2][0, u], mc, w.grid, w.block, "elu1", norm)
        for b in range(w.n_blocks):
            sel = blk == b
            err = orc.relative_max_error(o[u][sel], want[sel])
            assert err <= TOL["bf16"], f"{norm}/{variant} unit {u} block {b} (scale {scales[b]:.0e}): {err:.3e}"


@pytest.mark.parametrize("case", ["v_1e-6", "v_1e3", "exp_k_to_20"])
def test_full_video_head_at_extremes(case):
    """One full-size video head (16x64x64 tokens, 512 blocks of 2x8x8) at
    each extreme, on the path the library picks for it."""
    fmap, kw = CASES[case]
    w = wl.WORKLOADS["video_16x64x64"].with_(batch=1, heads=1)
    vals, dev = rescaled(w, **kw)
    for norm in ("divisive", "none"):
        err = check(w, vals, dev, norm, "auto", fmap)
        assert err <= TOL["bf16"], f"{case}/{norm}: rel err {err:.3e}"
