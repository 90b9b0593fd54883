"""The accuracy bar for the GPU path against the fp64 oracle.

For each output tensor separately (o, and the final state hT), with x* the
oracle's fp64 result on the same (bf16 / fp32) inputs:

    relative L2 error   ||x - x*||_2 / ||x*||_2                    <= 1e-2
    max absolute error  max_i ( |x_i - x*_i| - r_i )               <= 2e-2 * RMS(x*)

r_i is the representation allowance of the output format: half a unit in the
last place of bf16 at the element's magnitude for o, which the interface fixes
to bf16, and 0 for the fp32 state.  Reason: bf16 keeps 8 significant bits, so
rounding even the exact result can move an element by up to 2^-8 of itself;
with max|o| / RMS(o) ~ 7.5 on the long workloads, the correctly rounded oracle
output alone misses the plain bound (2.1e-2 and 2.2e-2 * RMS measured on the
B2-H16-T32768 and B1-H32-T262144 input distributions).  The allowance removes
exactly that representational step and bounds everything else.
"""

from __future__ import annotations

import numpy as np

REL_L2 = 1e-2
MAX_ABS_OVER_RMS = 2e-2


def half_ulp_bf16(x) -> np.ndarray:
    """Half the bf16 spacing at |x| (0 for x == 0)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126.0)  # bf16 subnormal spacing is constant below 2^-126
    return np.where(ax > 0, np.exp2(e - 8.0), 0.0)


def error_report(x, ref, bf16_output: bool = False) -> dict:
    """Relative L2 error, the plain max abs error, the max abs error beyond the
    output rounding allowance, and the RMS of ref."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    diff = np.abs(x - ref)
    nref = np.linalg.norm(ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    rel = float(np.linalg.norm(diff) / nref) if nref > 0 else float(np.linalg.norm(diff))
    plain = float(np.max(diff)) if diff.size else 0.0
    if bf16_output:
        diff = diff - half_ulp_bf16(np.maximum(np.abs(x), np.abs(ref)))
    excess = float(np.max(diff)) if diff.size else 0.0
    return {"rel_l2": rel, "max_abs": plain, "max_abs_excess": excess, "rms": rms}


def errors(x, ref, bf16_output: bool = False):
    """Returns (relative L2 error, max excess abs error, RMS of ref)."""
    r = error_report(x, ref, bf16_output)
    return r["rel_l2"], r["max_abs_excess"], r["rms"]


# Every comparison made in this process, for the run's closing summary: the plain
# max abs error is reported beside the one the bar applies to.
RECORDS: list = []


def assert_close(x, ref, what: str = "", bf16_output: bool = False) -> dict:
    xa = np.asarray(x, dtype=np.float64)
    assert np.all(np.isfinite(xa)), f"{what}: non-finite values"
    r = error_report(xa, ref, bf16_output)
    rel, maxabs, rms = r["rel_l2"], r["max_abs_excess"], r["rms"]
    RECORDS.append(dict(r, what=what, bf16_output=bf16_output))
    plain = (f"plain max abs {r['max_abs']:.3e} = {r['max_abs'] / rms:.3e} RMS"
             if rms > 0 else f"plain max abs {r['max_abs']:.3e}")
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2} ({plain})"
    bound = MAX_ABS_OVER_RMS * rms
    assert maxabs <= bound or (rms == 0.0 and maxabs <= 0.0), (
        f"{what}: max abs error beyond the output rounding {maxabs:.3e} > "
        f"{MAX_ABS_OVER_RMS} * RMS ({bound:.3e}); {plain}")
    return r
