"""Shared helpers of the GPU tests: seeded inputs on the device and the
tolerances of the parity checks.

Tolerances (fixed numerically for the two input precisions):
  * fp32 inputs: max |gpu - ref| / max |ref| <= 1e-4 (normwise relative);
  * bf16 inputs (fp32 accumulation and state): max |gpu - ref| <= 2e-2 and
    RMS(gpu - ref) <= 1e-2, measured after GroupNorm.
"""
import numpy as np
import torch

from linear_recurrent_sequence_gb300 import synth

TOL_F32_REL = 1e-4
TOL_BF16_MAX = 2e-2
TOL_BF16_RMS = 1e-2


def seeded(seed, name, shape, dtype, std=1.0, device="cuda"):
    """(device tensor, exact float64 numpy values) of a seeded tensor."""
    store, x64 = synth.tensor(seed, name, shape, dtype, std)
    if dtype == "bf16":
        t = torch.from_numpy(store.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(store)
    return t.to(device), x64


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_f32(got, ref, what=""):
    err = np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30)
    assert err <= TOL_F32_REL, f"{what}: normwise rel err {err:.3e} > {TOL_F32_REL}"
    return err


def check_bf16(got, ref, what=""):
    d = np.abs(got - ref)
    mx, rms = float(d.max()), float(np.sqrt((d ** 2).mean()))
    assert mx <= TOL_BF16_MAX and rms <= TOL_BF16_RMS, \
        f"{what}: max abs {mx:.3e} (<= {TOL_BF16_MAX}), rms {rms:.3e} (<= {TOL_BF16_RMS})"
    return mx, rms
