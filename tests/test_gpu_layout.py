"""Token-major tensors ([B, N, H, d], MHLA_LAYOUT_BNHD) on every path: the
results must be bitwise those of the head-major layout ([B, H, N, d]) on the
same values -- the kernels run the same tiles in the same order, only the
addresses differ -- and hence carry the head-major path's oracle parity."""

import numpy as np
import pytest

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


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _tok(t):
    return t.permute(0, 2, 1, 3).contiguous()


CASES = [("deit_t", "simt"), ("deit_t", "multipass"), ("deit_t", "fused"), ("tiny_f32", "simt"),
         ("wan_21x30x50", "multipass"), ("seq_32k", "multipass"), ("video_16x64x64", "multipass")]


@pytest.mark.parametrize("norm", ["divisive", "mala"])
@pytest.mark.parametrize("name,variant", CASES)
def test_forward_token_major_is_bitwise_head_major(name, variant, norm):
    import torch
    w = wl.WORKLOADS[name]
    if name in ("wan_21x30x50", "seq_32k", "video_16x64x64"):
        w = w.with_(batch=2, heads=3)
    vals, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    a = mb.mhla_forward(q, k, v, mc, w.grid, w.block, norm=norm, variant=variant)
    b = mb.mhla_forward(_tok(q), _tok(k), _tok(v), mc, w.grid, w.block, norm=norm, variant=variant, layout="bnhd")
    torch.cuda.synchronize()
    assert torch.equal(_bits(_tok(b)), _bits(a))
    o = download(a).reshape(w.units, w.n_tokens, w.head_dim)
    want = orc.mhla_head64(vals[0][0, 0], vals[1][0, 0], vals[2][0, 0], wl.make_mc(w), w.grid, w.block, "elu1", norm)
    assert orc.relative_max_error(o[0], want) <= TOL[w.dtype]


@pytest.mark.parametrize("variant", ["auto", "simt"])
def test_backward_token_major_is_bitwise_head_major(variant):
    import torch
    w = wl.WORKLOADS["deit_t"].with_(batch=4)
    _, dev = wl.all_inputs(w)
    _, gdev = wl.output_grad(w)
    q, k, v = upload(w, dev)
    (g,) = upload(w, [gdev])
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    a = mb.mhla_backward(q, k, v, mc, g, w.grid, w.block, variant=variant)
    b = mb.mhla_backward(_tok(q), _tok(k), _tok(v), mc, _tok(g), w.grid, w.block, variant=variant, layout="bnhd")
    torch.cuda.synchronize()
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(_bits(_tok(y)), _bits(x))
    assert torch.equal(a[3], b[3])


def test_causal_token_major_is_bitwise_head_major():
    import torch
    w = wl.random_small(51, (1, 1, 512), (1, 1, 64), 64, 2, 3, "bf16")
    _, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    a = mb.mhla_forward(q, k, v, mc, w.grid, w.block, causal=True)
    b = mb.mhla_forward(_tok(q), _tok(k), _tok(v), mc, w.grid, w.block, causal=True, layout="bnhd")
    torch.cuda.synchronize()
    assert torch.equal(_bits(_tok(b)), _bits(a))


def test_host_entry_token_major():
    # the pipelined host entry splits the problem into groups of whole batches
    import torch
    w = wl.WORKLOADS["image_64x64"]
    _, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    a = mb.mhla_forward(q, k, v, mc, w.grid, w.block)
    hq, hk, hv = (_tok(t).cpu().pin_memory() for t in (q, k, v))
    hmc = mc.cpu().pin_memory()
    out = torch.empty_like(hq).pin_memory()
    mb.mhla_forward_host(hq, hk, hv, hmc, w.grid, w.block, out=out, layout="bnhd")
    torch.cuda.synchronize()
    assert torch.equal(_bits(_tok(out.cuda())), _bits(a))
