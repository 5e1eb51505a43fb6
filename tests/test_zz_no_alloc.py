"""The allocation-free entry point (mhla_forward_noalloc), for callers that
cannot allocate device memory when they call: its scratch is a static device
array inside the library.  Checked through the C ABI against mhla_forward on
two calls in a row (the second call finds the first call's leftovers in the
shared array).  Collected last so that a run stopping at the first failure
has run every other test already."""

import ctypes

import pytest

from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

from helpers import TOL, download, upload

pytestmark = pytest.mark.gpu

CASES = [
    wl.WORKLOADS["deit_t"],                                   # tensor-core path
    wl.WORKLOADS["tiny_f32"],                                 # CUDA-core path
    wl.random_small(31, (1, 16, 16), (1, 4, 4), 64, 2, 2, "bf16").with_(norm="mala"),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from token_level_head_phi_gb300 import build
    build.build()
    mb.load()


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.name}-{w.norm}")
def test_noalloc_matches_forward_twice(w):
    torch = pytest.importorskip("torch")
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype, "elu1", w.norm)
    assert mb.mhla_workspace_bytes(p) <= 32 << 20
    vals, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    ref = download(mb.mhla_forward(q, k, v, mc, w.grid, w.block, norm=w.norm))
    stream = torch.cuda.current_stream().cuda_stream
    lib = mb.load()
    for call in range(2):
        out = torch.empty_like(q)
        st = lib.mhla_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), ctypes.byref(p),
                                      out.data_ptr(), stream)
        assert st == mb.MHLA_OK, mb.mhla_status_string(st)
        torch.cuda.synchronize()
        got = download(out)
        assert orc.relative_max_error(got, ref) <= TOL[w.dtype], f"call {call}"
    code, detail = mb.mhla_device_status()
    assert code == 0, (code, detail)


def test_noalloc_rejects_problems_beyond_its_scratch():
    torch = pytest.importorskip("torch")
    w = wl.WORKLOADS["video_16x64x64"]
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype)
    assert mb.mhla_workspace_bytes(p) > 32 << 20
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = mb.load().mhla_forward_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), ctypes.byref(p),
                                        x.data_ptr() + 16, torch.cuda.current_stream().cuda_stream)
    assert st == mb.MHLA_ERR_WORKSPACE
