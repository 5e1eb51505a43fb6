"""Shared helpers of the GPU parity tests: upload seeded inputs, run the
library through its C ABI (ctypes binding), fetch results, run the oracle on
the same values."""

from __future__ import annotations

import numpy as np

from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import binding as mb
from token_level_head_phi_gb300 import workloads as wl

TOL = {"bf16": 5e-3, "f32": 1e-5}


def torch_mod():
    import torch
    return torch


def upload(w: wl.Workload, dev_arrays, device="cuda"):
    torch = torch_mod()
    out = []
    for a in dev_arrays:
        t = torch.from_numpy(np.ascontiguousarray(a))
        if w.dtype == "bf16":
            t = t.view(torch.bfloat16)
        out.append(t.to(device))
    return out


def download(t) -> np.ndarray:
    torch = torch_mod()
    if t.dtype == torch.bfloat16:
        bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
        return wl.bf16_bits_to_f32(bits).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def run_gpu(w: wl.Workload, tensors, mc: np.ndarray, norm: str, variant: str = "auto",
            fmap: str = "elu1", out=None):
    torch = torch_mod()
    q, k, v = tensors
    mct = torch.from_numpy(np.ascontiguousarray(mc, dtype=np.float32)).cuda()
    o = mb.mhla_forward(q, k, v, mct, w.grid, w.block, norm=norm, feature_map=fmap, variant=variant, out=out)
    torch.cuda.synchronize()
    code, detail = mb.mhla_device_status()
    assert code == 0, f"device status {code} (detail {detail})"
    return o


def oracle_unit(w: wl.Workload, vals, unit: int, mc, norm: str, fmap: str = "elu1") -> np.ndarray:
    b, h = divmod(unit, w.heads)
    return orc.mhla_head64(vals[0][b, h], vals[1][b, h], vals[2][b, h], mc, w.grid, w.block, fmap, norm)


def parity(w: wl.Workload, norm: str, variant: str = "auto", units=None, mc=None, fmap: str = "elu1",
           inputs=None):
    """Run the GPU on every unit, the oracle on `units` (all if None);
    returns the worst max|gpu - oracle| / max|oracle| over those units."""
    vals, dev = inputs if inputs is not None else wl.all_inputs(w)
    mc = wl.make_mc(w) if mc is None else mc
    tensors = upload(w, dev)
    o = download(run_gpu(w, tensors, mc, norm, variant, fmap)).reshape(w.units, w.n_tokens, w.head_dim)
    units = range(w.units) if units is None else units
    worst = 0.0
    for u in units:
        want = oracle_unit(w, vals, u, mc, norm, fmap)
        assert np.all(np.isfinite(o[u])), f"non-finite output in unit {u}"
        worst = max(worst, orc.relative_max_error(o[u], want))
    return worst
