"""Per-head mixing matrices (Mc [H, M, M], one per head, shared over the
batch) on every path: parity with the oracle's per-head entry points, and
H identical copies bitwise equal to one shared matrix."""

import numpy as np
import pytest

from oracle import mhla_backward_oracle as orb
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


def _mcs(w):
    # one locality-biased matrix per head (different noise seeds)
    return np.stack([wl.make_mc(w.with_(seed=w.seed + 101 * h)) for h in range(w.heads)]).astype(np.float32)


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


CASES = [("deit_t", "multipass"), ("deit_t", "simt"), ("tiny_f32", "simt"), ("seq_32k", "multipass"),
         ("video_16x64x64", "multipass"), ("wan_21x30x50", "multipass")]


@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("name,variant", CASES)
def test_forward_per_head_mc(name, variant, norm):
    import torch
    w = wl.WORKLOADS[name]
    if w.n_tokens > 4096:
        w = w.with_(batch=2, heads=3)
    if name == "tiny_f32":
        w = w.with_(heads=3)
    vals, dev = wl.all_inputs(w)
    mcs = _mcs(w)
    q, k, v = upload(w, dev)
    o = mb.mhla_forward(q, k, v, torch.from_numpy(mcs).cuda(), w.grid, w.block, norm=norm, variant=variant)
    torch.cuda.synchronize()
    code, detail = mb.mhla_device_status()
    assert code == 0, (code, detail)
    o = download(o)
    for b, h in ((0, 0), (w.batch - 1, w.heads - 1), (0, w.heads - 1)):
        want = orc.mhla_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mcs[h], w.grid, w.block, "elu1", norm)
        assert orc.relative_max_error(o[b, h], want) <= TOL[w.dtype], (b, h)


@pytest.mark.parametrize("variant", ["multipass", "simt"])
def test_identical_copies_equal_shared_mc(variant):
    import torch
    w = wl.WORKLOADS["deit_t"]
    _, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    a = mb.mhla_forward(q, k, v, mc, w.grid, w.block, variant=variant)
    b = mb.mhla_forward(q, k, v, mc.expand(w.heads, -1, -1).contiguous(), w.grid, w.block, variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(_bits(a), _bits(b))


@pytest.mark.parametrize("norm", ["divisive", "mala"])
def test_causal_per_head_mc(norm):
    import torch
    w = wl.random_small(61, (1, 1, 512), (1, 1, 64), 64, 2, 3, "bf16")
    vals, dev = wl.all_inputs(w)
    mcs = _mcs(w)
    q, k, v = upload(w, dev)
    o = download(mb.mhla_forward(q, k, v, torch.from_numpy(mcs).cuda(), w.grid, w.block, norm=norm, causal=True))
    want = occ.mhla_causal_forward64(vals[0], vals[1], vals[2], mcs, w.grid, w.block, norm=norm)
    for b in range(2):
        for h in range(3):
            assert orc.relative_max_error(o[b, h], want[b, h]) <= TOL["bf16"]


@pytest.mark.parametrize("variant", ["auto", "simt"])
@pytest.mark.parametrize("norm", ["divisive", "mala"])
def test_backward_per_head_mc(variant, norm):
    import torch
    w = wl.WORKLOADS["deit_t"].with_(batch=4)
    vals, dev = wl.all_inputs(w)
    gvals, gdev = wl.output_grad(w)
    mcs = _mcs(w)
    q, k, v = upload(w, dev)
    (g,) = upload(w, [gdev])
    got = mb.mhla_backward(q, k, v, torch.from_numpy(mcs).cuda(), g, w.grid, w.block, norm=norm, variant=variant)
    torch.cuda.synchronize()
    want = orb.mhla_backward64(vals[0], vals[1], vals[2], mcs.astype(np.float64), w.grid, w.block, gvals, "elu1",
                               norm)
    for x, y in zip(got[:3], want[:3]):
        assert orc.relative_max_error(download(x), y) <= 5e-3
    dmc = got[3].cpu().numpy().astype(np.float64)
    assert dmc.shape == (w.heads, w.n_blocks, w.n_blocks)
    tol = 2e-3 if variant == "auto" else 5e-4
    assert orc.relative_max_error(dmc, want[3]) <= tol


def test_host_entry_per_head_mc():
    import torch
    w = wl.WORKLOADS["image_64x64"]
    _, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mcs = torch.from_numpy(_mcs(w))
    a = mb.mhla_forward(q, k, v, mcs.cuda(), w.grid, w.block)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    out = torch.empty_like(hq).pin_memory()
    mb.mhla_forward_host(hq, hk, hv, mcs.pin_memory(), w.grid, w.block, out=out)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out.cuda()), _bits(a))
