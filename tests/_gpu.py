"""Helpers for the GPU parity tests: device buffers, host copies, tolerances."""
import numpy as np
import torch

import nvfp4_precision_moe_gb300 as nv

DEV = "cuda:0"


def lib():
    return nv.load(build=True)


def to_dev_bf16(t_cpu_bf16):
    return t_cpu_bf16.to(DEV)


def u16(t):
    """device/host BF16 tensor -> numpy uint16 bit patterns"""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_from_u16(a, dev=DEV):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def rel_err(y, ref):
    """max_i |y_i - ref_i| / max(|ref_i|, rms of ref's row): the GEMM parity
    metric (cancellation near zero is measured against the row's scale)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True)) + 1e-300
    den = np.maximum(np.abs(ref), rms)
    return float((np.abs(y - ref) / den).max())


def zeros(shape, dtype):
    return torch.zeros(shape, dtype=dtype, device=DEV)


def status_ok(st):
    v = int(st.item())
    assert v == 0, nv.STATUS.get(v, v)
