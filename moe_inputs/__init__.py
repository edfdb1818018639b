"""Seeded synthetic inputs for the MoE layer, shared by the CUDA path's tests/bench and the oracle.

Host tensors come from the numpy twin (``host.py``); device tensors from the CUDA twin
(``csrc/gen.cu``, built into ``libmoe_inputs.so``).  Both implement the same counter-based
recipe and are bit-identical, which ``tests/test_inputs_gpu.py`` checks elementwise.

Layer inputs (row-major, names follow the layer's notation):
  x          [T][d]          N(0, 1)
  w_router   [E][d]          N(0, 1/d)     (row e scores expert e)
  w_gate_up  [E][2F][d]      N(0, 1/d)     (per expert: F gate rows, then F up rows)
  w_down     [E][d][F]       N(0, 1/F)
  bias       [E]   fp32      U(-b, b)      (sigmoid configs; selection only)
  sh_gate_up [2Fs][d]        N(0, 1/d)     (shared expert, if Fs > 0)
  sh_down    [d][Fs]         N(0, 1/Fs)
Zipf-skewed configs additionally set x[:, 0] = 1 and w_router[:, 0] = the per-expert
offsets from ``host.zipf_offsets``, so the linear gate itself adds the offset to every
token's logits (no extra operator in the layer).
"""
import ctypes
import os

import numpy as np

from . import configs, host
from .configs import (TID_BIAS, TID_SH_DOWN, TID_SH_GATE_UP, TID_W_DOWN, TID_W_GATE_UP,
                      TID_W_ROUTER, TID_X)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_inputs.so")

# name -> (tensor id, shape fn, fan-in fn); std = 1/sqrt(fan_in) (x uses std 1)
_SPECS = {
    "x": (TID_X, lambda c: (c["T"], c["d"]), lambda c: 1),
    "w_router": (TID_W_ROUTER, lambda c: (c["E"], c["d"]), lambda c: c["d"]),
    "w_gate_up": (TID_W_GATE_UP, lambda c: (c["E"], 2 * c["F"], c["d"]), lambda c: c["d"]),
    "w_down": (TID_W_DOWN, lambda c: (c["E"], c["d"], c["F"]), lambda c: c["F"]),
    "sh_gate_up": (TID_SH_GATE_UP, lambda c: (2 * c["Fs"], c["d"]), lambda c: c["d"]),
    "sh_down": (TID_SH_DOWN, lambda c: (c["d"], c["Fs"]), lambda c: c["Fs"]),
}


def std_of(cfg, name):
    return 1.0 / np.sqrt(float(_SPECS[name][2](cfg)))


def shape_of(cfg, name):
    if name == "bias":
        return (cfg["E"],)
    return _SPECS[name][1](cfg)


def tensor_names(cfg):
    names = ["x", "w_router", "w_gate_up", "w_down"]
    if cfg["bias_range"] > 0:
        names.append("bias")
    if cfg["Fs"] > 0:
        names += ["sh_gate_up", "sh_down"]
    return names


def zipf(cfg):
    z = cfg["zipf"]
    return host.zipf_offsets(cfg["E"], cfg["seed"], z["s"], z["scale"])


def _patch_value(cfg, v):
    """fp32 value -> stored element (bf16 bits or fp32)."""
    v = np.asarray(v, dtype=np.float32)
    return host.f32_to_bf16_bits(v) if cfg["dtype"] == "bf16" else v


def host_tensor(cfg, name, lead=None):
    """Host copy of an input tensor; ``lead`` selects rows of the leading dimension."""
    cfg = configs.get(cfg)
    if name == "bias":
        idx = np.arange(cfg["E"], dtype=np.uint64) if lead is None else np.asarray(lead, np.uint64)
        return host.uniform_f32(idx, cfg["seed"], TID_BIAS, -cfg["bias_range"], cfg["bias_range"])
    tid = _SPECS[name][0]
    shape = shape_of(cfg, name)
    inner = int(np.prod(shape[1:]))
    lead_idx = np.arange(shape[0]) if lead is None else np.asarray(lead, dtype=np.int64)
    flat = (lead_idx.astype(np.uint64)[:, None] * np.uint64(inner)
            + np.arange(inner, dtype=np.uint64)[None, :]).ravel()
    out = host.normal(flat, cfg["seed"], tid, std_of(cfg, name), cfg["dtype"])
    out = out.reshape((len(lead_idx),) + tuple(shape[1:]))
    if cfg["zipf"] is not None and name in ("x", "w_router"):
        if name == "x":
            out[:, 0] = _patch_value(cfg, 1.0)
        else:
            off, _ = zipf(cfg)
            out[:, 0] = _patch_value(cfg, off[lead_idx])
    return out


def host_inputs(cfg):
    cfg = configs.get(cfg)
    return {n: host_tensor(cfg, n) for n in tensor_names(cfg)}


def as_float64(cfg, arr):
    """Stored elements (bf16 bits or fp32) -> exact fp64 values."""
    if configs.get(cfg)["dtype"] == "bf16" and arr.dtype == np.uint16:
        return host.bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float64)


# ---------------------------------------------------------------------------------------
# device twin
_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
        l = ctypes.CDLL(LIB_PATH)
        l.moegen_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                         ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                         ctypes.c_void_p]
        l.moegen_fill_normal.restype = ctypes.c_int
        l.moegen_fill_uniform.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_void_p]
        l.moegen_fill_uniform.restype = ctypes.c_int
        _lib = l
    return _lib


def device_tensor(cfg, name, device="cuda"):
    """Generate one input tensor directly in device memory (torch tensor)."""
    import torch
    cfg = configs.get(cfg)
    stream = torch.cuda.current_stream(device).cuda_stream
    if name == "bias":
        t = torch.empty(cfg["E"], dtype=torch.float32, device=device)
        rc = lib().moegen_fill_uniform(t.data_ptr(), t.numel(), cfg["seed"], TID_BIAS,
                                       -cfg["bias_range"], cfg["bias_range"], stream)
        if rc != 0:
            raise RuntimeError(f"moegen_fill_uniform failed: {rc}")
        return t
    tid = _SPECS[name][0]
    dt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    t = torch.empty(shape_of(cfg, name), dtype=dt, device=device)
    rc = lib().moegen_fill_normal(t.data_ptr(), 1 if cfg["dtype"] == "bf16" else 0, t.numel(),
                                  cfg["seed"], tid, float(std_of(cfg, name)), stream)
    if rc != 0:
        raise RuntimeError(f"moegen_fill_normal failed: {rc}")
    if cfg["zipf"] is not None and name in ("x", "w_router"):
        if name == "x":
            t[:, 0] = 1.0
        else:
            off, _ = zipf(cfg)
            t[:, 0] = torch.from_numpy(off).to(device=device, dtype=dt)
    return t


def device_inputs(cfg, device="cuda"):
    cfg = configs.get(cfg)
    return {n: device_tensor(cfg, n, device) for n in tensor_names(cfg)}


def upload(cfg, arrays, device="cuda"):
    """Host arrays (bf16 bits / fp32) -> device torch tensors, byte-identical."""
    import torch
    cfg = configs.get(cfg)
    out = {}
    for n, a in arrays.items():
        if a.dtype == np.uint16:
            out[n] = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
        else:
            out[n] = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return out
