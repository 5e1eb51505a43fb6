"""The allocation-free entry point (mhla_forward_noalloc), for callers that
cannot allocate device memory when they call: its scratch is a static device
array inside the library.  Checked through the C ABI against mhla_forward and
against the float64 oracle on two calls in a row (the second call finds the
first call's leftovers in the shared array), on the tensor-core path, the
CUDA-core path, the fused launch (whose progress counters live in that array
and must start from zero on every call) and the causal form; and checked to
allocate nothing (the default memory pool and torch's allocator are unchanged
across a call).  Collected last so that a run stopping at the first failure
has run every other test already."""

import ctypes

import numpy as np
import pytest

from oracle import mhla_causal_oracle as occ
from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

from helpers import TOL, download, upload

pytestmark = pytest.mark.gpu

# (workload, variant, causal)
CASES = [
    (wl.WORKLOADS["deit_t"], "auto", False),                                   # tensor cores, fp16 records
    (wl.WORKLOADS["tiny_f32"], "auto", False),                                 # CUDA cores
    (wl.random_small(31, (1, 16, 16), (1, 4, 4), 64, 2, 2, "bf16").with_(norm="mala"), "auto", False),
    (wl.random_small(32, (1, 16, 16), (1, 4, 8), 64, 2, 3, "bf16"), "fused", False),
    (wl.random_small(33, (1, 1, 1024), (1, 1, 256), 64, 1, 2, "bf16"), "auto", True),   # causal, two chunks per block
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from token_level_head_phi_gb300 import build
    build.build()
    mb.load()


def _noalloc(w, tensors, mc, variant, causal, out):
    torch = pytest.importorskip("torch")
    q, k, v = tensors
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype, "elu1", w.norm, variant, causal)
    st = mb.load().mhla_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), ctypes.byref(p),
                                        out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == mb.MHLA_OK, mb.mhla_status_string(st)
    torch.cuda.synchronize()


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}-{c[0].norm}-{c[1]}{'-causal' if c[2] else ''}")
def test_noalloc_matches_forward_and_oracle_twice(case):
    torch = pytest.importorskip("torch")
    w, variant, causal = case
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype, "elu1", w.norm, variant, causal)
    assert mb.mhla_workspace_bytes(p) <= 32 << 20
    vals, dev = wl.all_inputs(w)
    tensors = upload(w, dev)
    mcn = wl.make_mc(w)
    mc = torch.from_numpy(mcn).cuda()
    ref = download(mb.mhla_forward(*tensors, mc, w.grid, w.block, norm=w.norm, variant=variant, causal=causal))
    for call in range(2):
        out = torch.empty_like(tensors[0])
        _noalloc(w, tensors, mc, variant, causal, out)
        got = download(out)
        assert orc.relative_max_error(got, ref) <= TOL[w.dtype], f"call {call}: differs from mhla_forward"
        o = got.reshape(w.units, w.n_tokens, w.head_dim)
        for u in (0, w.units - 1):
            b, h = divmod(u, w.heads)
            args = (vals[0][b, h], vals[1][b, h], vals[2][b, h], mcn, w.grid, w.block, "elu1", w.norm)
            want = occ.mhla_causal_head64(*args) if causal else orc.mhla_head64(*args)
            assert orc.relative_max_error(o[u], want) <= TOL[w.dtype], f"call {call} unit {u}: differs from the oracle"
    code, detail = mb.mhla_device_status()
    assert code == 0, (code, detail)


def _cudart():
    for name in ("libcudart.so", "libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


def test_noalloc_allocates_nothing():
    """Across a call (after a first one), the device's default memory pool --
    where stream-ordered allocations come from -- neither uses nor reserves
    more memory, even transiently (its usage high-water mark, reset before
    the call, stays at the current usage), and torch's allocator holds the
    same bytes."""
    torch = pytest.importorskip("torch")
    rt = _cudart()
    if rt is None:
        pytest.skip("the CUDA runtime library cannot be opened to read the memory pool")
    w = wl.WORKLOADS["deit_t"]
    _, dev = wl.all_inputs(w)
    tensors = upload(w, dev)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    out = torch.empty_like(tensors[0])
    _noalloc(w, tensors, mc, "auto", False, out)
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), torch.cuda.current_device()) == 0

    def attr(a):
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, a, ctypes.byref(v)) == 0
        return v.value

    RESERVED, USED, USED_HIGH = 0x5, 0x7, 0x8   # cudaMemPoolAttr values
    zero = ctypes.c_uint64(0)
    assert rt.cudaMemPoolSetAttribute(pool, USED_HIGH, ctypes.byref(zero)) == 0   # high-water mark := current
    before = (attr(RESERVED), attr(USED), torch.cuda.memory_allocated())
    _noalloc(w, tensors, mc, "auto", False, out)
    after = (attr(RESERVED), attr(USED), torch.cuda.memory_allocated())
    assert after == before, (before, after)
    assert attr(USED_HIGH) == after[1], "a transient stream-ordered allocation happened inside the call"


def test_noalloc_rejects_problems_beyond_its_scratch():
    torch = pytest.importorskip("torch")
    w = wl.WORKLOADS["video_16x64x64"]
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype)
    assert mb.mhla_workspace_bytes(p) > 32 << 20
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    st = mb.load().mhla_forward_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), ctypes.byref(p),
                                        x.data_ptr() + 16, torch.cuda.current_stream().cuda_stream)
    assert st == mb.MHLA_ERR_WORKSPACE
