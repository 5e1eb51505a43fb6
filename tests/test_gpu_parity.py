"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Measure: max|gpu - oracle| / max|oracle| per (batch, head) unit, at most 5e-3
for bf16 inputs/outputs with float32 accumulation and 1e-5 in float32 mode.
Full-size workloads compare every unit the oracle finishes in seconds and a
sample of units otherwise; edge cases cover ragged blocks, every head
dimension, a single block, Mc rows with zeros, non-square and 3D grids, every
norm and both feature maps.
"""

import zlib

import numpy as np
import pytest

from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

from helpers import TOL, download, parity, run_gpu, upload

pytestmark = pytest.mark.gpu

VARIANTS = ["simt", "multipass", "fused"]

FULL = {  # workload -> units the oracle checks (None = all)
    "tiny_f32": None,
    "deit_t": None,
    "image_64x64": None,
    "video_16x64x64": [0, 17, 31],
    "seq_32k": [0, 33, 63],
    "seq_32k_mala": [0, 63],
    "seq_32k_m1": [0, 40],
    "seq_32k_m1_mala": [1, 62],
    "wan_21x30x50": [0, 23],
}


def _tc_supported(dtype, d):
    return dtype == "bf16" and d == 64


def _skip_unsupported(variant, dtype, d):
    if variant in ("multipass", "fused") and not _tc_supported(dtype, d):
        pytest.skip("tensor-core path covers bf16 with d = 64")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from token_level_head_phi_gb300 import build
    build.build()
    mb.load()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", list(FULL))
def test_workload_parity(name, variant):
    w = wl.WORKLOADS[name]
    _skip_unsupported(variant, w.dtype, w.head_dim)
    err = parity(w, w.norm, variant, units=FULL[name])
    assert err <= TOL[w.dtype], f"{name}/{variant}: rel err {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("name", ["tiny_f32", "deit_t"])
def test_norms(name, norm, variant):
    w = wl.WORKLOADS[name]
    _skip_unsupported(variant, w.dtype, w.head_dim)
    err = parity(w, norm, variant, units=[0, w.units - 1])
    assert err <= TOL[w.dtype], f"{name}/{norm}/{variant}: rel err {err:.3e}"


EDGE = [
    # grid, block, d, dtype, batch, heads
    ((1, 14, 14), (1, 7, 7), 64, "bf16", 1, 2),        # ragged 49-token blocks
    ((1, 10, 12), (1, 5, 4), 32, "f32", 2, 1),         # non-square blocks, d=32
    ((3, 8, 8), (3, 4, 8), 16, "f32", 1, 3),           # 3D, bt = T, d=16
    ((4, 6, 10), (2, 3, 5), 128, "bf16", 1, 1),        # 3D ragged, d=128
    ((1, 1, 1000), (1, 1, 1000), 64, "bf16", 2, 2),    # one block, N not a multiple of 64
    ((1, 1, 3000), (1, 1, 1500), 64, "f32", 1, 1),     # two long blocks split into pieces
    ((1, 1, 4100), (1, 1, 41), 64, "bf16", 1, 1),      # M=100 odd blocks
    ((1, 9, 1), (1, 3, 1), 64, "bf16", 1, 1),          # column grid
    ((2, 2, 2), (1, 1, 1), 16, "f32", 1, 1),           # one token per block
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("norm", ["divisive", "mala"])
@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}-{c[3]}")
def test_edge_shapes(case, norm, variant):
    grid, block, d, dtype, batch, heads = case
    _skip_unsupported(variant, dtype, d)
    w = wl.random_small(zlib.crc32(repr(case).encode()) % 10000, grid, block, d, batch, heads, dtype)
    err = parity(w, norm, variant)
    assert err <= TOL[dtype], f"{case}/{norm}: rel err {err:.3e}"


LARGE_M_CASES = [
    # grid, block, heads: more than 128 query blocks, so the fp16 mixing takes
    # the streaming tensor-core kernel (256 query blocks per tile)
    ((1, 1, 2304), (1, 1, 16), 3),      # M = 144: one tile of 256 query blocks, 112 of them padding; Q % 64 = 16
    ((1, 1, 8192), (1, 1, 32), 2),      # M = 256: one full tile
    ((1, 1, 4160), (1, 1, 8), 1),       # M = 520: three 256-block tiles, the last with 8 rows
    ((1, 96, 96), (1, 6, 6), 2),        # 2D, M = 256, 36-token blocks
    ((4, 48, 48), (2, 4, 4), 1),        # 3D, M = 288
]


@pytest.mark.parametrize("norm", ["divisive", "none"])
@pytest.mark.parametrize("case", LARGE_M_CASES, ids=lambda c: f"{c[0]}-{c[1]}-h{c[2]}")
def test_large_m_mixing_shapes(case, norm):
    grid, block, heads = case
    w = wl.random_small(zlib.crc32(repr(case).encode()) % 10000, grid, block, 64, 1, heads, "bf16")
    assert w.n_blocks > 128
    err = parity(w, norm, "multipass")
    assert err <= TOL["bf16"], f"{case}/{norm}: rel err {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
def test_mc_with_zero_entries(variant):
    w = wl.random_small(5, (1, 16, 16), (1, 4, 4), 64, 2, 2, "bf16")
    M = w.n_blocks
    rng = np.random.default_rng(3)
    mc = rng.uniform(0, 1, (M, M)) * (rng.uniform(0, 1, (M, M)) < 0.3)
    np.fill_diagonal(mc, 1.0)
    mc = (mc / mc.sum(1, keepdims=True)).astype(np.float32)
    for norm in ("divisive", "mala", "none"):
        err = parity(w, norm, variant, mc=mc)
        assert err <= TOL["bf16"], f"{norm}: {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
def test_linear_decay_mc_and_identity_map(variant):
    dtype = "f32" if variant == "simt" else "bf16"
    w = wl.random_small(8, (1, 12, 12), (1, 4, 4), 64, 1, 2, dtype, mc="linear_decay")
    vals, dev = wl.all_inputs(w)
    vals = [np.abs(a) + 0.1 for a in vals]  # positive features for phi(x) = x
    if dtype == "bf16":
        pairs = [wl.round_to_bf16(a) for a in vals]
        dev = [b for b, _ in pairs]
        vals = [v for _, v in pairs]
    else:
        dev = [a.astype(np.float32) for a in vals]
    err = parity(w, "divisive", variant, fmap="identity", inputs=(vals, dev))
    assert err <= TOL[dtype]


@pytest.mark.parametrize("variant", VARIANTS)
def test_output_guard_regions_untouched(variant):
    torch = pytest.importorskip("torch")
    w = wl.random_small(9, (1, 14, 14), (1, 7, 7), 64, 2, 3, "bf16")
    vals, dev = wl.all_inputs(w)
    tensors = upload(w, dev)
    n = w.units * w.n_tokens * w.head_dim
    pad = 4096
    big = torch.full((n + 2 * pad,), 12345.0, dtype=torch.bfloat16, device="cuda")
    out = big[pad:pad + n].view(w.batch, w.heads, w.n_tokens, w.head_dim)
    run_gpu(w, tensors, wl.make_mc(w), "divisive", variant, out=out)
    assert torch.all(big[:pad] == 12345.0) and torch.all(big[pad + n:] == 12345.0)
    o = download(out).reshape(w.units, w.n_tokens, w.head_dim)
    mc = wl.make_mc(w)
    for u in range(w.units):
        b, h = divmod(u, w.heads)
        want = orc.mhla_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block)
        assert orc.relative_max_error(o[u], want) <= TOL["bf16"]


def test_host_entry_matches_device_entry():
    torch = pytest.importorskip("torch")
    w = wl.WORKLOADS["deit_t"]
    vals, dev = wl.all_inputs(w)
    mc = wl.make_mc(w)
    tensors = upload(w, dev)
    d_out = download(run_gpu(w, tensors, mc, "divisive"))
    host = [torch.from_numpy(a).view(torch.bfloat16).pin_memory() for a in dev]
    h_out = torch.empty_like(host[0]).pin_memory()
    mb.mhla_forward_host(*host, torch.from_numpy(mc), w.grid, w.block, out=h_out)
    np.testing.assert_array_equal(download(h_out), d_out)


def test_workspace_allocated_by_library():
    torch = pytest.importorskip("torch")
    import ctypes
    w = wl.WORKLOADS["tiny_f32"]
    vals, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mc = torch.from_numpy(wl.make_mc(w)).cuda()
    out = torch.empty_like(q)
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, "f32")
    st = mb.mhla_forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), p, out.data_ptr(), 0, 0,
                             torch.cuda.current_stream().cuda_stream)
    assert st == mb.MHLA_OK
    torch.cuda.synchronize()
    want = orc.mhla_head64(vals[0][0, 0], vals[1][0, 0], vals[2][0, 0], wl.make_mc(w), w.grid, w.block)
    assert orc.relative_max_error(download(out)[0, 0], want) <= TOL["f32"]
    del ctypes


def test_phase_events_recorded():
    torch = pytest.importorskip("torch")
    w = wl.WORKLOADS["image_64x64"]
    vals, dev = wl.all_inputs(w)
    tensors = upload(w, dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(mb.NUM_PHASE_EVENTS)]
    mb.mhla_set_phase_events(ev)
    try:
        run_gpu(w, tensors, wl.make_mc(w), "divisive")
    finally:
        mb.mhla_set_phase_events(None)
    times = [ev[0].elapsed_time(ev[i]) for i in range(1, mb.NUM_PHASE_EVENTS)]
    assert all(t >= 0 for t in times) and times == sorted(times)


def _run_variant(w, tensors, mc, norm, variant):
    torch = pytest.importorskip("torch")
    o = run_gpu(w, tensors, mc, norm, variant)
    return o.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("name", ["seq_32k_mala", "image_64x64"])
def test_fused_bitwise_equals_multipass_mala(name):
    """Under MALA both launches run the same split-precision arithmetic in
    the same order on the tensor cores: the results are bit for bit the same.
    (DIVISIVE and NONE mix fp16 records in the multi-pass launch and split
    records in the fused one, and the multi-pass launch mixes 16 blocks or
    fewer on the CUDA cores; test_workload_parity checks every one of them
    against the oracle.)"""
    w = wl.WORKLOADS[name].with_(norm="mala")
    vals, dev = wl.all_inputs(w)
    tensors = upload(w, dev)
    mc = wl.make_mc(w)
    a = _run_variant(w, tensors, mc, w.norm, "multipass")
    b = _run_variant(w, tensors, mc, w.norm, "fused")
    np.testing.assert_array_equal(a, b)


# CTA counts of the (summary, mixing, output) groups: one CTA each, lopsided
# splits either way, and far more streaming than mixing CTAs
GROUP_SPLITS = ["1,1,1", "7,1,2", "1,9,1", "2,3,40", "60,2,60"]


@pytest.mark.parametrize("groups", GROUP_SPLITS)
@pytest.mark.parametrize("norm", ["divisive", "mala"])
def test_fused_group_splits(groups, norm, monkeypatch):
    """However the SMs are split between the groups, the fused launch gives
    the same bits (its default split is the reference) and matches the oracle."""
    w = wl.random_small(77, (1, 16, 16), (1, 4, 8), 64, 4, 6, "bf16")
    vals, dev = wl.all_inputs(w)
    tensors = upload(w, dev)
    mc = wl.make_mc(w)
    monkeypatch.delenv("MHLA_FUSED_GROUPS", raising=False)
    ref = _run_variant(w, tensors, mc, norm, "fused")
    monkeypatch.setenv("MHLA_FUSED_GROUPS", groups)
    got = _run_variant(w, tensors, mc, norm, "fused")
    np.testing.assert_array_equal(ref, got)
    o = download(run_gpu(w, tensors, mc, norm, "fused")).reshape(w.units, w.n_tokens, w.head_dim)
    for u in (0, w.units - 1):
        b, h = divmod(u, w.heads)
        want = orc.mhla_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block, "elu1", norm)
        assert orc.relative_max_error(o[u], want) <= TOL["bf16"]


def test_fused_wait_expires_and_reports():
    """A wait on another CTA group that can never end (the output group asks
    for one mixing signal too many) expires after a short limit, every CTA
    stops, the device status reads MHLA_ERR_DEVICE_TIMEOUT, and the next call
    runs normally."""
    torch = pytest.importorskip("torch")
    w = wl.random_small(31, (1, 16, 16), (1, 4, 8), 64, 2, 3, "bf16")
    vals, dev = wl.all_inputs(w)
    q, k, v = upload(w, dev)
    mc = wl.make_mc(w)
    mct = torch.from_numpy(mc).cuda()
    out = torch.zeros_like(q)
    mb.mhla_set_debug(mb.DEBUG_FLOW_WAIT_NS, 20_000_000)
    mb.mhla_set_debug(mb.DEBUG_FLOW_STALL, 1)
    try:
        mb.mhla_forward(q, k, v, mct, w.grid, w.block, variant="fused", out=out)
        code, detail = mb.mhla_device_status()
    finally:
        mb.mhla_set_debug(mb.DEBUG_FLOW_STALL, 0)
        mb.mhla_set_debug(mb.DEBUG_FLOW_WAIT_NS, 0)
    assert code == mb.MHLA_ERR_DEVICE_TIMEOUT, (code, detail)
    o = download(run_gpu(w, (q, k, v), mc, "divisive", "fused")).reshape(w.units, w.n_tokens, w.head_dim)
    for u in (0, w.units - 1):
        assert orc.relative_max_error(o[u], oracle_unit_divisive(w, vals, u, mc)) <= TOL["bf16"]


def oracle_unit_divisive(w, vals, unit, mc):
    b, h = divmod(unit, w.heads)
    return orc.mhla_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block)


@pytest.mark.parametrize("name", ["seq_32k", "video_16x64x64"])
def test_host_entry_pipelined_matches_device_entry(name):
    """Large problems go through the host entry point in head groups whose
    copies overlap the kernels; the result is the device entry's, bit for bit."""
    torch = pytest.importorskip("torch")
    w = wl.WORKLOADS[name]
    vals, dev = wl.all_inputs(w)
    mc = wl.make_mc(w)
    tensors = upload(w, dev)
    d_out = run_gpu(w, tensors, mc, w.norm).view(torch.int16).cpu().numpy()
    del tensors
    host = [torch.from_numpy(a).view(torch.bfloat16).pin_memory() for a in dev]
    h_out = torch.empty_like(host[0]).pin_memory()
    mb.mhla_forward_host(*host, torch.from_numpy(mc), w.grid, w.block, norm=w.norm, out=h_out)
    np.testing.assert_array_equal(h_out.view(torch.int16).numpy(), d_out)


# ---------------------------------------------------------------- feature maps

@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("norm", ["divisive", "none", "mala"])
@pytest.mark.parametrize("fmap", ["relu", "exp"])
@pytest.mark.parametrize("name", ["tiny_f32", "deit_t"])
def test_relu_and_exp_maps(name, fmap, norm, variant):
    w = wl.WORKLOADS[name]
    _skip_unsupported(variant, w.dtype, w.head_dim)
    err = parity(w, norm, variant, units=[0, w.units - 1], fmap=fmap)
    assert err <= TOL[w.dtype], f"{name}/{fmap}/{norm}/{variant}: rel err {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
def test_relu_maps_on_full_video_head(variant):
    w = wl.WORKLOADS["video_16x64x64"].with_(batch=1, heads=2)
    err = parity(w, "divisive", variant, fmap="relu")
    assert err <= TOL[w.dtype], f"{variant}: rel err {err:.3e}"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("norm", ["divisive", "mala"])
def test_zero_denominator_rows_are_zero(norm, variant):
    # ReLU features: a query with every entry negative has phi(q) = 0, and a
    # query whose only positive feature no key has sees s = 0 too; both
    # outputs are 0, every other output matches the oracle
    w = wl.random_small(31, (1, 14, 14), (1, 7, 7), 64, 1, 2, "bf16")
    vals, _ = wl.all_inputs(w)
    q, k, v = (np.array(a) for a in vals)
    q[:, :, 3, :] = -np.abs(q[:, :, 3, :]) - 0.25
    k[:, :, :, 0] = -np.abs(k[:, :, :, 0]) - 0.25
    q[:, :, 17, :] = -np.abs(q[:, :, 17, :]) - 0.25
    q[:, :, 17, 0] = 1.5
    pairs = [wl.round_to_bf16(a) for a in (q, k, v)]
    dev = [b for b, _ in pairs]
    vals = [x for _, x in pairs]
    mc = wl.make_mc(w)
    o = download(run_gpu(w, upload(w, dev), mc, norm, variant, "relu")).reshape(w.units, w.n_tokens, w.head_dim)
    assert np.all(np.isfinite(o))
    assert np.all(o[:, 3] == 0.0) and np.all(o[:, 17] == 0.0)
    for u in range(w.units):
        want = orc.mhla_head64(vals[0][0, u], vals[1][0, u], vals[2][0, u], mc, w.grid, w.block, "relu", norm)
        assert orc.relative_max_error(o[u], want) <= TOL["bf16"]
