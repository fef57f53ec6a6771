"""Shared helpers of the GPU tests: seeded inputs on the device and the
tolerances of the parity checks.

Tolerances (fixed numerically for the two input precisions):
  * fp32 inputs: max |gpu - ref| / max |ref| <= 1e-4 (normwise relative);
  * bf16 inputs (fp32 accumulation and state): max |gpu - ref| <= 2e-2 and
    RMS(gpu - ref) <= 1e-2, measured after GroupNorm.  For outputs stored in
    bf16 the max-abs bound applies to the error beyond the half ulp of the
    storage rounding; fp32-output runs of the same workloads are checked
    with no allowance.
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


def bf16_half_ulp(x):
    """Half the spacing of bfloat16 numbers at |x| (8 significant bits): the
    largest error of rounding x to bf16 (normal range)."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8.0)


def check_bf16(got, ref, what="", spread=None):
    """Max abs and RMS of got - ref after GroupNorm.  When `got` was stored
    in bf16 (every value representable in bf16), the max-abs check measures
    the arithmetic error: it allows, on top of the tolerance, the half ulp of
    rounding the exact result to bf16 for storage (for a GroupNorm output of
    |y| >= 8 that rounding alone can reach 2^-5, above the tolerance).
    `spread` (optional, one value per output row): the exact function's own
    sensitivity to rounding its operands (operand_sensitivity); each row's
    max-abs bound is widened by twice it.  The RMS check has no allowance."""
    d = np.abs(got - ref)
    stored_bf16 = bool(np.all(np.asarray(got, np.float32) == bf16_round(got)))
    e = np.maximum(d - bf16_half_ulp(ref), 0.0) if stored_bf16 else d
    if spread is not None:
        e = np.maximum(e - 2.0 * np.asarray(spread)[..., None], 0.0)
    mx, rms = float(e.max()), float(np.sqrt((d ** 2).mean()))
    where = np.unravel_index(int(np.argmax(e)), e.shape)
    assert mx <= TOL_BF16_MAX and rms <= TOL_BF16_RMS, \
        f"{what}: max abs {mx:.3e} at {tuple(int(i) for i in where)} " \
        f"(<= {TOL_BF16_MAX}{' beyond bf16 storage' if stored_bf16 else ''}), " \
        f"rms {rms:.3e} (<= {TOL_BF16_RMS})"
    return mx, rms


# Unit roundoff of the fp16 operands of the tensor-core path (11 significant
# bits, round to nearest).
FP16_U = 2.0 ** -11


def operand_sensitivity(run, q64, k64, seed=0):
    """Per output row (the last axis reduced), how far the exact float64
    result moves when q and k are perturbed by relative errors of up to the
    fp16 unit roundoff, as the tensor-core path rounds them: `run(q, k)`
    returns the oracle's output.  Where a row's result is that sensitive
    (the first tokens of a sequence, whose few score terms can cancel), no
    implementation with fp16 operands can be closer to the exact value than
    about this much."""
    g = np.random.default_rng(seed)
    ref = run(q64, k64)
    qp = q64 * (1.0 + FP16_U * g.uniform(-1.0, 1.0, q64.shape))
    kp = k64 * (1.0 + FP16_U * g.uniform(-1.0, 1.0, k64.shape))
    return np.abs(run(qp, kp) - ref).max(axis=-1)


def bf16_round(x):
    """float64 values rounded as the GPU path stores them in bf16 (through
    float32, then to nearest even)."""
    return synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(np.asarray(x, np.float32)))


def split_ill_conditioned(ref, ref_rounded, axis_token=-2, tol=TOL_BF16_MAX):
    """Boolean mask over the token axis of the tokens on which the float64
    result changes by more than `tol` when the inputs of its steps are
    rounded to bf16 where the GPU path stores them: there the function itself
    amplifies the unavoidable input rounding (GroupNorm of a row whose
    variance is near its epsilon, after a cancelling dot product), so no
    bf16 implementation can match the unrounded result."""
    d = np.abs(ref - ref_rounded)
    axes = tuple(i for i in range(d.ndim) if i != d.ndim + axis_token)
    return d.max(axis=axes) > tol
