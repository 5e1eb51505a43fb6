"""ctypes binding of libmhla.so (include/mhla.h), same names as the C ABI.

Only argument marshalling happens here: tensors are checked for device,
dtype, shape and contiguity, their ``data_ptr()`` and the current CUDA
stream are handed to the library, and a non-OK status raises
:class:`MhlaError`.  Every step of the forward pass runs in the library's
kernels; there is no fallback of any kind -- if ``libmhla.so`` is missing the
first call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmhla.so")

MHLA_OK = 0
MHLA_ERR_INVALID_ARG = 1
MHLA_ERR_UNSUPPORTED = 2
MHLA_ERR_WORKSPACE = 3
MHLA_ERR_CUDA = 4
MHLA_ERR_DEVICE_TIMEOUT = 5
MHLA_ERR_OVERFLOW = 6

DTYPE_BF16 = 0
DTYPE_F32 = 1
FEATURE_ELU1 = 0
FEATURE_IDENTITY = 1
FEATURE_RELU = 2
FEATURE_EXP = 3
NORM_DIVISIVE = 0
NORM_MALA = 1
NORM_NONE = 2
VARIANT_AUTO = 0
VARIANT_SIMT = 1
VARIANT_MULTIPASS = 2
VARIANT_FUSED = 3
NUM_PHASE_EVENTS = 6
NUM_BWD_PHASE_EVENTS = 6

NORMS = {"divisive": NORM_DIVISIVE, "mala": NORM_MALA, "none": NORM_NONE}
FEATURE_MAPS = {"elu1": FEATURE_ELU1, "identity": FEATURE_IDENTITY, "relu": FEATURE_RELU, "exp": FEATURE_EXP}
VARIANTS = {"auto": VARIANT_AUTO, "simt": VARIANT_SIMT, "multipass": VARIANT_MULTIPASS, "fused": VARIANT_FUSED}
DTYPES = {"bf16": DTYPE_BF16, "f32": DTYPE_F32}
LAYOUT_BHND = 0
LAYOUT_BNHD = 1
LAYOUTS = {"bhnd": LAYOUT_BHND, "bnhd": LAYOUT_BNHD}


class MhlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib_or_none()
        text = lib.mhla_status_string(status).decode() if lib else f"status {status}"
        detail = lib.mhla_last_error_string().decode() if (lib and status == MHLA_ERR_CUDA) else ""
        super().__init__(f"{where}: {text}" + (f" ({detail})" if detail else ""))
        self.status = status


class MhlaParams(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("grid", ctypes.c_int * 3), ("block", ctypes.c_int * 3),
        ("dtype", ctypes.c_int), ("feature_map", ctypes.c_int), ("norm", ctypes.c_int),
        ("variant", ctypes.c_int), ("causal", ctypes.c_int), ("layout", ctypes.c_int),
        ("mc_per_head", ctypes.c_int),
    ]


class MhlaPlanInfo(ctypes.Structure):
    _fields_ = [
        ("n_tokens", ctypes.c_int), ("n_blocks", ctypes.c_int), ("block_tokens", ctypes.c_int),
        ("variant", ctypes.c_int), ("kernels_per_call", ctypes.c_int), ("summary_splits", ctypes.c_int),
        ("workspace_bytes", ctypes.c_size_t),
    ]


_LIB = None

# (name, restype, argtypes) of every entry point in include/mhla.h
SIGNATURES = [
    ("mhla_plan", ctypes.c_int, [ctypes.POINTER(MhlaParams), ctypes.POINTER(MhlaPlanInfo)]),
    ("mhla_workspace_bytes", ctypes.c_int, [ctypes.POINTER(MhlaParams), ctypes.POINTER(ctypes.c_size_t)]),
    ("mhla_forward", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.POINTER(MhlaParams), ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_size_t, ctypes.c_void_p]),
    ("mhla_forward_noalloc", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.POINTER(MhlaParams), ctypes.c_void_p, ctypes.c_void_p]),
    ("mhla_host_buffer_bytes", ctypes.c_int, [ctypes.POINTER(MhlaParams), ctypes.POINTER(ctypes.c_size_t)]),
    ("mhla_forward_host", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.POINTER(MhlaParams), ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]),
    ("mhla_device_status", ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    ("mhla_set_phase_events", ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
    ("mhla_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("mhla_last_error_string", ctypes.c_char_p, []),
    ("mhla_abi_version", ctypes.c_int, []),
    ("mhla_set_debug", ctypes.c_int, [ctypes.c_int, ctypes.c_longlong]),
    ("mhla_set_backward_phase_events", ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
    ("mhla_backward_workspace_bytes", ctypes.c_int, [ctypes.POINTER(MhlaParams), ctypes.POINTER(ctypes.c_size_t)]),
    ("mhla_backward", ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.POINTER(MhlaParams)] + [ctypes.c_void_p] * 5
     + [ctypes.c_size_t, ctypes.c_void_p]),
]


def _lib_or_none():
    return _LIB


def load(path: Optional[str] = None):
    """Load libmhla.so (once) and declare every entry point's signature."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m token_level_head_phi_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, restype, argtypes in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = restype
        fn.argtypes = argtypes
    _LIB = lib
    return lib


def _check(status: int, where: str):
    if status != MHLA_OK:
        raise MhlaError(status, where)


def make_params(batch: int, heads: int, head_dim: int, grid: Sequence[int], block: Sequence[int],
                dtype: str = "bf16", feature_map: str = "elu1", norm: str = "divisive",
                variant: str = "auto", causal: bool = False, layout: str = "bhnd",
                mc_per_head: bool = False) -> MhlaParams:
    p = MhlaParams()
    p.batch, p.heads, p.head_dim = int(batch), int(heads), int(head_dim)
    for i in range(3):
        p.grid[i] = int(grid[i])
        p.block[i] = int(block[i])
    p.dtype = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    p.feature_map = FEATURE_MAPS[feature_map] if isinstance(feature_map, str) else int(feature_map)
    p.norm = NORMS[norm] if isinstance(norm, str) else int(norm)
    p.variant = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    p.causal = int(causal)
    p.layout = LAYOUTS[layout] if isinstance(layout, str) else int(layout)
    p.mc_per_head = int(mc_per_head)
    return p


def mhla_plan(p: MhlaParams) -> MhlaPlanInfo:
    info = MhlaPlanInfo()
    _check(load().mhla_plan(ctypes.byref(p), ctypes.byref(info)), "mhla_plan")
    return info


def mhla_workspace_bytes(p: MhlaParams) -> int:
    n = ctypes.c_size_t(0)
    _check(load().mhla_workspace_bytes(ctypes.byref(p), ctypes.byref(n)), "mhla_workspace_bytes")
    return n.value


def mhla_host_buffer_bytes(p: MhlaParams) -> int:
    n = ctypes.c_size_t(0)
    _check(load().mhla_host_buffer_bytes(ctypes.byref(p), ctypes.byref(n)), "mhla_host_buffer_bytes")
    return n.value


def _torch_dtype_name(t) -> str:
    import torch
    if t.dtype == torch.bfloat16:
        return "bf16"
    if t.dtype == torch.float32:
        return "f32"
    raise TypeError(f"unsupported dtype {t.dtype}; MHLA takes bfloat16 or float32")


def _mc_per_head(mc, p) -> int:
    """1 when mc is [H, M, M] (one matrix per head), 0 when it is [M, M]."""
    if mc.dim() == 3:
        if mc.shape[0] != p.heads:
            raise ValueError(f"per-head mc must be [H={p.heads}, M, M], got {tuple(mc.shape)}")
        return 1
    if mc.dim() != 2:
        raise ValueError("mc must be [M, M] or [H, M, M]")
    return 0


def _params_for(q, grid, block, feature_map, norm, variant, causal=False, layout="bhnd") -> MhlaParams:
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d] (layout 'bhnd') or [B, N, H, d] (layout 'bnhd')")
    if layout == "bnhd":
        B, N, H, d = q.shape
    else:
        B, H, N, d = q.shape
    if grid[0] * grid[1] * grid[2] != N:
        raise ValueError(f"grid {tuple(grid)} has {grid[0] * grid[1] * grid[2]} tokens, tensors have {N}")
    return make_params(B, H, d, grid, block, _torch_dtype_name(q), feature_map, norm, variant, causal, layout)


def mhla_forward(q, k, v, mc, grid, block, norm: str = "divisive", feature_map: str = "elu1",
                 variant: str = "auto", out=None, workspace=None, stream=None, causal: bool = False,
                 layout: str = "bhnd"):
    """MHLA forward on CUDA tensors [B, H, N, d]; returns ``out``.

    ``mc`` is a float32 [M, M] CUDA tensor.  ``out`` and ``workspace`` are
    allocated with torch when not given.  The call is enqueued on ``stream``
    (default: torch's current stream) and does not synchronise.
    """
    import torch
    p = _params_for(q, grid, block, feature_map, norm, variant, causal, layout)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor shaped and typed like q")
    if not mc.is_cuda or mc.dtype != torch.float32 or not mc.is_contiguous():
        raise ValueError("mc must be a contiguous float32 CUDA tensor")
    p.mc_per_head = _mc_per_head(mc, p)
    if out is None:
        out = torch.empty_like(q)
    elif not out.is_cuda or not out.is_contiguous() or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    need = mhla_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    status = load().mhla_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), ctypes.byref(p),
                                 out.data_ptr(), workspace.data_ptr(), ws_bytes, handle)
    _check(status, "mhla_forward")
    return out


def mhla_backward_workspace_bytes(p: MhlaParams) -> int:
    n = ctypes.c_size_t(0)
    _check(load().mhla_backward_workspace_bytes(ctypes.byref(p), ctypes.byref(n)), "mhla_backward_workspace_bytes")
    return n.value


def mhla_backward(q, k, v, mc, dout, grid, block, norm: str = "divisive", feature_map: str = "elu1",
                  dq=None, dk=None, dv=None, dmc=None, workspace=None, stream=None, variant: str = "auto",
                  layout: str = "bhnd", causal: bool = False):
    """Gradients of sum(dout * mhla_forward(q, k, v, mc)): returns (dq, dk, dv, dmc).

    dq, dk, dv are shaped and typed like q; dmc is float32 [M, M] (summed
    over every batch and head).  Outputs and workspace are allocated with
    torch when not given; enqueued on ``stream`` without synchronising.
    ``variant``: "auto" (tensor cores for bf16 with d = 64, else float32 CUDA
    cores) or "simt" (float32 CUDA cores).  ``causal``: the block-ordered
    causal form (float32 CUDA cores).
    """
    import torch
    p = _params_for(q, grid, block, feature_map, norm, variant, causal, layout)
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        if not t.is_cuda or not t.is_contiguous() or t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor shaped and typed like q")
    if not mc.is_cuda or mc.dtype != torch.float32 or not mc.is_contiguous():
        raise ValueError("mc must be a contiguous float32 CUDA tensor")
    p.mc_per_head = _mc_per_head(mc, p)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if not t.is_cuda or not t.is_contiguous() or t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor shaped and typed like q")
    if dmc is None:
        dmc = torch.empty_like(mc)
    elif not dmc.is_cuda or dmc.dtype != torch.float32 or not dmc.is_contiguous() or dmc.shape != mc.shape:
        raise ValueError("dmc must be a contiguous float32 CUDA tensor shaped like mc")
    need = mhla_backward_workspace_bytes(p)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    status = load().mhla_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), dout.data_ptr(),
                                  ctypes.byref(p), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dmc.data_ptr(),
                                  workspace.data_ptr(), ws_bytes, handle)
    _check(status, "mhla_backward")
    return dq, dk, dv, dmc


def mhla_forward_raw(q_ptr: int, k_ptr: int, v_ptr: int, mc_ptr: int, p: MhlaParams, out_ptr: int,
                     ws_ptr: int, ws_bytes: int, stream_handle: int) -> int:
    """Direct call with raw device pointers; returns the status code."""
    return load().mhla_forward(q_ptr, k_ptr, v_ptr, mc_ptr, ctypes.byref(p), out_ptr, ws_ptr, ws_bytes,
                               stream_handle)


def mhla_forward_noalloc(q, k, v, mc, grid, block, norm: str = "divisive", feature_map: str = "elu1",
                         variant: str = "auto", out=None, stream=None, layout: str = "bhnd"):
    """mhla_forward without any device allocation by the library: its scratch
    is a static 32 MiB device array (see include/mhla.h).  For callers that
    cannot allocate at call time; ``out`` must be given by such callers (when
    it is None this wrapper allocates it with torch, for convenience)."""
    import torch
    p = _params_for(q, grid, block, feature_map, norm, variant, False, layout)
    p.mc_per_head = _mc_per_head(mc, p)
    if out is None:
        out = torch.empty_like(q)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    status = load().mhla_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), ctypes.byref(p),
                                         out.data_ptr(), handle)
    _check(status, "mhla_forward_noalloc")
    return out


def mhla_forward_host(q, k, v, mc, grid, block, norm: str = "divisive", feature_map: str = "elu1",
                      variant: str = "auto", out=None, dev_buffer=None, stream=None, causal: bool = False,
                      layout: str = "bhnd"):
    """End-to-end call on CPU tensors (pinned for asynchronous copies).

    Copies the inputs into ``dev_buffer`` (a CUDA uint8 tensor of at least
    ``mhla_host_buffer_bytes`` bytes), runs the forward pass and copies the
    result back into ``out``; returns when ``out`` is complete.
    """
    import torch
    p = _params_for(q, grid, block, feature_map, norm, variant, causal, layout)
    p.mc_per_head = _mc_per_head(mc, p)
    for name, t in (("q", q), ("k", k), ("v", v), ("mc", mc)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    if out is None:
        out = torch.empty_like(q)
    need = mhla_host_buffer_bytes(p)
    if dev_buffer is None:
        dev_buffer = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    if stream is None:
        stream = torch.cuda.current_stream(dev_buffer.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    status = load().mhla_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), ctypes.byref(p),
                                      out.data_ptr(), dev_buffer.data_ptr(),
                                      dev_buffer.numel() * dev_buffer.element_size(), handle)
    _check(status, "mhla_forward_host")
    return out


def mhla_device_status():
    """(code, detail) of the device error word; blocks until the device is idle."""
    code, detail = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().mhla_device_status(ctypes.byref(code), ctypes.byref(detail)), "mhla_device_status")
    return code.value, detail.value


def mhla_set_phase_events(events) -> None:
    """Install (list of NUM_PHASE_EVENTS torch.cuda.Event) or clear (None) the phase-timing hook."""
    if events is None:
        _check(load().mhla_set_phase_events(None, 0), "mhla_set_phase_events")
        return
    for e in events:  # torch creates the CUDA event on its first record
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().mhla_set_phase_events(arr, len(events)), "mhla_set_phase_events")


def mhla_set_backward_phase_events(events) -> None:
    """The same hook for mhla_backward (NUM_BWD_PHASE_EVENTS events, or None)."""
    if events is None:
        _check(load().mhla_set_backward_phase_events(None, 0), "mhla_set_backward_phase_events")
        return
    for e in events:
        if not e.cuda_event:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(load().mhla_set_backward_phase_events(arr, len(events)), "mhla_set_backward_phase_events")


def mhla_backward_raw(q_ptr: int, k_ptr: int, v_ptr: int, mc_ptr: int, dout_ptr: int, p: MhlaParams, dq_ptr: int,
                      dk_ptr: int, dv_ptr: int, dmc_ptr: int, ws_ptr: int, ws_bytes: int, stream_handle: int) -> int:
    """Direct call with raw device pointers; returns the status code."""
    return load().mhla_backward(q_ptr, k_ptr, v_ptr, mc_ptr, dout_ptr, ctypes.byref(p), dq_ptr, dk_ptr, dv_ptr,
                                dmc_ptr, ws_ptr, ws_bytes, stream_handle)


def mhla_status_string(status: int) -> str:
    return load().mhla_status_string(status).decode()


DEBUG_FLOW_WAIT_NS = 1
DEBUG_FLOW_STALL = 2


def mhla_set_debug(option: int, value: int) -> None:
    """Testing hooks of the fused launch's waits (see mhla.h)."""
    _check(load().mhla_set_debug(int(option), int(value)), "mhla_set_debug")


def mhla_abi_version() -> int:
    return load().mhla_abi_version()
