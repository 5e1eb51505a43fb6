"""CPU checks of the C ABI: the library builds, loads, exports every symbol
include/mhla.h declares, and validates arguments on the host before touching
the device.  No call here reaches a CUDA runtime function."""

import ctypes
import os
import re

import pytest

from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import build as mbuild
from token_level_head_phi_gb300 import workloads as wl

HEADER = os.path.join(mbuild.INCLUDE, "mhla.h")


@pytest.fixture(scope="session")
def lib():
    mbuild.build()
    return mb.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mhla_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = header_functions()
    assert "mhla_forward" in names and "mhla_workspace_bytes" in names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"{name} missing from libmhla.so"


def test_binding_declares_every_header_function():
    bound = {s[0] for s in mb.SIGNATURES}
    assert set(header_functions()) == bound


def test_abi_version_and_strings(lib):
    assert mb.mhla_abi_version() == 3
    for s in range(7):
        assert mb.mhla_status_string(s).startswith("MHLA")
    assert "unknown" in mb.mhla_status_string(42)


def _params(w, **kw):
    opts = dict(dtype=w.dtype, norm=w.norm)
    opts.update(kw)
    return mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, **opts)


@pytest.mark.parametrize("name", sorted(wl.WORKLOADS))
def test_plan_matches_workload(lib, name):
    w = wl.WORKLOADS[name]
    info = mb.mhla_plan(_params(w, variant="simt"))
    assert info.n_tokens == w.n_tokens
    assert info.n_blocks == w.n_blocks
    assert info.block_tokens == w.block_tokens
    assert info.variant == mb.VARIANT_SIMT
    assert info.kernels_per_call >= 1
    d, R = w.head_dim, w.head_dim ** 2 + 2 * w.head_dim
    stack = 4 * w.units * w.n_blocks * info.summary_splits * R
    mixed = 4 * w.units * w.n_blocks * R
    assert info.workspace_bytes >= stack + mixed
    assert mb.mhla_workspace_bytes(_params(w, variant="simt")) == info.workspace_bytes


BAD = [
    dict(head_dim=48),
    dict(head_dim=0),
    dict(grid=(1, 15, 14)),      # 15 not divisible by 7
    dict(block=(1, 0, 7)),
    dict(grid=(0, 14, 14)),
    dict(batch=-1),
    dict(dtype=7),
    dict(feature_map=4),
    dict(feature_map=-1),
    dict(norm=9),
    dict(variant=11),
    dict(layout=2),
    dict(causal=3),
    dict(mc_per_head=2),
]


@pytest.mark.parametrize("bad", BAD)
def test_invalid_params_rejected(lib, bad):
    w = wl.WORKLOADS["deit_t"]
    args = dict(batch=w.batch, heads=w.heads, head_dim=w.head_dim, grid=w.grid, block=w.block)
    opts = dict(dtype=w.dtype, norm="divisive", feature_map="elu1", variant="auto")
    for k, v in bad.items():
        (args if k in args else opts)[k] = v
    p = mb.make_params(args["batch"], args["heads"], args["head_dim"], args["grid"], args["block"], **opts)
    info = mb.MhlaPlanInfo()
    assert lib.mhla_plan(ctypes.byref(p), ctypes.byref(info)) == mb.MHLA_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert lib.mhla_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == mb.MHLA_ERR_INVALID_ARG
    # forward rejects the same parameters before looking at any pointer
    assert lib.mhla_forward(None, None, None, None, ctypes.byref(p), None, None, 0, None) == \
        mb.MHLA_ERR_INVALID_ARG


def test_null_params_rejected(lib):
    assert lib.mhla_forward(None, None, None, None, None, None, None, 0, None) == mb.MHLA_ERR_INVALID_ARG
    assert lib.mhla_workspace_bytes(None, None) == mb.MHLA_ERR_INVALID_ARG


def test_empty_problem_is_noop(lib):
    w = wl.WORKLOADS["deit_t"]
    for batch, heads in ((0, 3), (4, 0)):
        p = mb.make_params(batch, heads, 64, w.grid, w.block)
        assert mb.mhla_workspace_bytes(p) == 0
        assert lib.mhla_forward(None, None, None, None, ctypes.byref(p), None, None, 0, None) == mb.MHLA_OK


FAKE = 1 << 40  # never dereferenced: validation fails first


def test_pointer_checks(lib):
    w = wl.WORKLOADS["deit_t"]
    p = _params(w)
    io = w.units * w.n_tokens * w.head_dim * 2
    q, k, v, mc, out, ws = FAKE, FAKE + 2 * io, FAKE + 4 * io, FAKE + 6 * io, FAKE + 8 * io, FAKE + 10 * io
    need = mb.mhla_workspace_bytes(p)
    f = lib.mhla_forward
    # null pointers
    assert f(None, k, v, mc, ctypes.byref(p), out, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, None, ctypes.byref(p), out, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, ctypes.byref(p), None, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    # misaligned tensors / workspace
    assert f(q + 2, k, v, mc, ctypes.byref(p), out, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc + 2, ctypes.byref(p), out, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, ctypes.byref(p), out + 8, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, ctypes.byref(p), out, ws + 16, need, None) == mb.MHLA_ERR_INVALID_ARG
    # output aliasing an input
    assert f(q, k, v, mc, ctypes.byref(p), q + 256, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    # workspace too small, or sized but null
    assert f(q, k, v, mc, ctypes.byref(p), out, ws, need - 1, None) == mb.MHLA_ERR_WORKSPACE
    assert f(q, k, v, mc, ctypes.byref(p), out, None, need, None) == mb.MHLA_ERR_INVALID_ARG


def test_host_entry_checks(lib):
    w = wl.WORKLOADS["tiny_f32"]
    p = _params(w)
    need = mb.mhla_host_buffer_bytes(p)
    io = w.units * w.n_tokens * w.head_dim * 4
    assert need >= 4 * io + mb.mhla_workspace_bytes(p)
    h = ctypes.create_string_buffer(io)
    f = lib.mhla_forward_host
    assert f(h, h, h, h, ctypes.byref(p), h, None, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(h, h, h, h, ctypes.byref(p), h, FAKE, need - 1, None) == mb.MHLA_ERR_WORKSPACE


def test_phase_event_hook_checks(lib):
    assert lib.mhla_set_phase_events(None, 0) == mb.MHLA_OK
    assert lib.mhla_set_phase_events(None, mb.NUM_PHASE_EVENTS) == mb.MHLA_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 3)(1, 2, 3)
    assert lib.mhla_set_phase_events(arr, 3) == mb.MHLA_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 4)(1, 2, None, 3)
    assert lib.mhla_set_phase_events(arr, 4) == mb.MHLA_ERR_INVALID_ARG
    assert lib.mhla_set_backward_phase_events(None, 0) == mb.MHLA_OK
    assert lib.mhla_set_backward_phase_events(None, mb.NUM_BWD_PHASE_EVENTS) == mb.MHLA_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 4)(1, 2, 3, 4)
    assert lib.mhla_set_backward_phase_events(arr, 4) == mb.MHLA_ERR_INVALID_ARG


def test_long_blocks_are_split(lib):
    w = wl.WORKLOADS["seq_32k_m1"]
    info = mb.mhla_plan(_params(w, variant="simt"))
    assert info.n_blocks == 1 and info.summary_splits > 1


def test_auto_picks_tensor_cores_for_bf16_d64(lib):
    w = wl.WORKLOADS["video_16x64x64"]
    assert mb.mhla_plan(_params(w)).variant == mb.VARIANT_MULTIPASS
    assert mb.mhla_plan(_params(wl.WORKLOADS["tiny_f32"])).variant == mb.VARIANT_SIMT
    p = mb.make_params(1, 1, 32, (1, 8, 8), (1, 4, 4), "bf16")
    assert mb.mhla_plan(p).variant == mb.VARIANT_SIMT


@pytest.mark.parametrize("variant", ["multipass", "fused"])
def test_tensor_core_variants_reject_unsupported(lib, variant):
    info = mb.MhlaPlanInfo()
    for dtype, d in (("f32", 64), ("bf16", 32), ("bf16", 128)):
        p = mb.make_params(1, 1, d, (1, 8, 8), (1, 4, 4), dtype, variant=variant)
        assert lib.mhla_plan(ctypes.byref(p), ctypes.byref(info)) == mb.MHLA_ERR_UNSUPPORTED


def test_multipass_splits_long_blocks(lib):
    w = wl.WORKLOADS["seq_32k_m1"]
    info = mb.mhla_plan(_params(w, variant="multipass"))
    assert info.summary_splits > 1
    assert mb.mhla_plan(_params(wl.WORKLOADS["video_16x64x64"], variant="multipass")).summary_splits == 1


@pytest.mark.parametrize("name", ["deit_t", "video_16x64x64", "seq_32k", "seq_32k_mala", "seq_32k_m1"])
def test_fused_plan(lib, name):
    """The fused launch is the prep kernel plus one cooperative kernel; it
    keeps split (bf16 high + low) records for every norm, in a ring that never
    needs more workspace than the multi-pass buffers of the same records
    (MALA's), and needs less once the heads outnumber the ring."""
    w = wl.WORKLOADS[name]
    fused = mb.mhla_plan(_params(w, variant="fused"))
    multi = mb.mhla_plan(_params(w, variant="multipass"))
    split = mb.mhla_plan(_params(w, variant="multipass", norm="mala"))
    assert fused.variant == mb.VARIANT_FUSED and fused.kernels_per_call == 2
    # fp16 records need the exponent-folding kernel unless the mixing of few
    # blocks (M <= 16) runs on the CUDA cores, which also needs no prep kernel
    small = w.n_blocks <= 16 and w.n_blocks * multi.summary_splits <= 256
    if w.norm == "mala":
        assert multi.kernels_per_call == 4
    else:
        assert multi.kernels_per_call == (3 if small else 5)
    assert fused.summary_splits == multi.summary_splits
    assert fused.workspace_bytes <= split.workspace_bytes + 3 * 4 * w.units + 256
    if name == "video_16x64x64":
        assert fused.workspace_bytes < multi.workspace_bytes / 4


def test_debug_options(lib):
    assert lib.mhla_set_debug(0, 0) == mb.MHLA_ERR_INVALID_ARG
    assert lib.mhla_set_debug(99, 1) == mb.MHLA_ERR_INVALID_ARG
    for opt in (mb.DEBUG_FLOW_WAIT_NS, mb.DEBUG_FLOW_STALL):
        assert lib.mhla_set_debug(opt, 5) == mb.MHLA_OK
        assert lib.mhla_set_debug(opt, 0) == mb.MHLA_OK


def test_backward_workspace_and_checks(lib):
    w = wl.WORKLOADS["deit_t"]
    p = _params(w)
    d, R = w.head_dim, w.head_dim ** 2 + 2 * w.head_dim
    info = mb.mhla_plan(_params(w, variant="simt"))
    rows = w.units * w.n_blocks * info.summary_splits
    need = mb.mhla_backward_workspace_bytes(p)
    # per-piece summaries and their gradients, mixed summaries and their gradients
    assert need >= 4 * (2 * rows * R + rows + 2 * w.units * w.n_blocks * R + w.n_blocks)
    # the tensor-core backward (bf16, d = 64) keeps its records as bf16 planes
    # besides; the CUDA-core one needs only the float32 records
    simt = mb.mhla_backward_workspace_bytes(_params(w, variant="simt"))
    assert simt >= 4 * (2 * rows * R + rows + 2 * w.units * w.n_blocks * R + w.n_blocks)
    assert need > simt
    io = w.units * w.n_tokens * d * 2
    q, k, v, dout = FAKE, FAKE + 2 * io, FAKE + 4 * io, FAKE + 6 * io
    mc, dq, dk, dv, dmc, ws = FAKE + 8 * io, FAKE + 10 * io, FAKE + 12 * io, FAKE + 14 * io, FAKE + 16 * io, \
        FAKE + 18 * io
    f = lib.mhla_backward
    P = ctypes.byref(p)
    assert f(q, k, v, mc, dout, None, dq, dk, dv, dmc, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, None, P, dq, dk, dv, dmc, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout, P, dq, dk, dv, None, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout + 2, P, dq, dk, dv, dmc, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout, P, dq, dk + 8, dv, dmc, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout, P, dq, dk, dv, dmc + 2, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    # gradients aliasing an input or each other
    assert f(q, k, v, mc, dout, P, q + 256, dk, dv, dmc, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout, P, dq, dq + 256, dv, dmc, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout, P, dq, dk, dv, dv + 256, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout, P, dq, dk, dv, mc, ws, need, None) == mb.MHLA_ERR_INVALID_ARG
    # workspace
    assert f(q, k, v, mc, dout, P, dq, dk, dv, dmc, ws, need - 1, None) == mb.MHLA_ERR_WORKSPACE
    assert f(q, k, v, mc, dout, P, dq, dk, dv, dmc, None, need, None) == mb.MHLA_ERR_INVALID_ARG
    assert f(q, k, v, mc, dout, P, dq, dk, dv, dmc, ws + 16, need, None) == mb.MHLA_ERR_INVALID_ARG
    # invalid shapes fail before any pointer is looked at; empty problems are no-ops
    bad = mb.make_params(1, 1, 48, w.grid, w.block)
    assert f(None, None, None, None, None, ctypes.byref(bad), None, None, None, None, None, 0, None) == \
        mb.MHLA_ERR_INVALID_ARG
    empty = mb.make_params(0, 3, 64, w.grid, w.block)
    assert mb.mhla_backward_workspace_bytes(empty) == 0
    assert f(None, None, None, None, None, ctypes.byref(empty), None, None, None, None, None, 0, None) == mb.MHLA_OK


def test_causal_plan_and_rejections(lib):
    w = wl.WORKLOADS["deit_t"]
    # bf16, d = 64, DIVISIVE: the tensor-core causal path (mask, prep, summary, mixing, output)
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, causal=True)
    info = mb.mhla_plan(p)
    assert info.variant == mb.VARIANT_MULTIPASS and info.kernels_per_call == 5
    # MALA and float32 take the CUDA-core causal kernels
    mala = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, norm="mala", causal=True)
    assert mb.mhla_plan(mala).variant == mb.VARIANT_SIMT
    f32 = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, dtype="f32", causal=True)
    info32 = mb.mhla_plan(f32)
    assert info32.variant == mb.VARIANT_SIMT and info32.kernels_per_call == 5
    for variant, norm in (("fused", "divisive"), ("multipass", "mala")):
        bad = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, norm=norm, variant=variant, causal=True)
        assert lib.mhla_plan(ctypes.byref(bad), ctypes.byref(mb.MhlaPlanInfo())) == mb.MHLA_ERR_UNSUPPORTED
    # the causal backward runs on the CUDA cores: AUTO and SIMT plan it,
    # the tensor-core variants are refused
    n = ctypes.c_size_t(0)
    assert lib.mhla_backward_workspace_bytes(ctypes.byref(p), ctypes.byref(n)) == mb.MHLA_OK and n.value > 0
    for variant in ("simt", "multipass", "fused"):
        bq = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, variant=variant, causal=True)
        want = mb.MHLA_OK if variant == "simt" else mb.MHLA_ERR_UNSUPPORTED
        assert lib.mhla_backward_workspace_bytes(ctypes.byref(bq), ctypes.byref(n)) == want
    p.causal = 2
    assert lib.mhla_plan(ctypes.byref(p), ctypes.byref(mb.MhlaPlanInfo())) == mb.MHLA_ERR_INVALID_ARG


def test_per_head_mc_plan(lib):
    w = wl.WORKLOADS["image_64x64"]
    shared = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block)
    per_head = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, mc_per_head=True)
    assert mb.mhla_workspace_bytes(per_head) > mb.mhla_workspace_bytes(shared)
    fused = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, variant="fused", mc_per_head=True)
    assert lib.mhla_plan(ctypes.byref(fused), ctypes.byref(mb.MhlaPlanInfo())) == mb.MHLA_ERR_UNSUPPORTED
