"""Helpers of the GPU parity tests: device copies, guarded outputs, tolerances.

Tolerances (the bars the build is held to):
* fp16-input leg: relative Frobenius error <= 2e-3 and max |err| <= 1e-2 * rms(ref);
* exact-fp32 leg (the FFMA GEMM and the GEMV): relative Frobenius <= 1e-5;
* standalone dequant: bit exact.
The reference is always the float64 oracle result (before its final f32
rounding), on the same seeded inputs.
"""

import numpy as np
import torch

F16_REL = 2e-3
F16_MAX_OVER_RMS = 1e-2
EXACT_REL = 1e-5
GUARD = 256                    # canary floats on each side of an output
CANARY_BITS = 0x7FC0DEAD       # a NaN payload nothing computes


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(rows, cols):
    """NaN-filled [rows][cols] f32 view with canary bands on both sides."""
    n = rows * cols
    buf = torch.full((n + 2 * GUARD,), 0, dtype=torch.int32, device="cuda")
    buf[:GUARD] = CANARY_BITS
    buf[GUARD + n:] = CANARY_BITS
    buf[GUARD:GUARD + n] = 0x7FC00000  # quiet NaN: untouched outputs show
    view = buf[GUARD:GUARD + n].view(torch.float32).view(rows, cols)
    return buf, view


def check_guards(buf, rows, cols):
    n = rows * cols
    head = buf[:GUARD].cpu().numpy()
    tail = buf[GUARD + n:].cpu().numpy()
    assert np.all(head == CANARY_BITS) and np.all(tail == CANARY_BITS), "write outside the output"


def errors(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(y)), "non-finite output (an element was not written?)"
    d = y - ref
    nref = np.linalg.norm(ref)
    rel = float(np.linalg.norm(d) / nref) if nref > 0 else float(np.linalg.norm(d))
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    mx = float(np.max(np.abs(d))) if d.size else 0.0
    return rel, mx, rms


def assert_f16_leg(y, ref):
    rel, mx, rms = errors(y, ref)
    assert rel <= F16_REL, f"rel-Frobenius {rel:.3e} > {F16_REL}"
    assert mx <= F16_MAX_OVER_RMS * rms, f"max|err| {mx:.3e} > 1e-2 * rms {rms:.3e}"
    return rel, mx / rms if rms else 0.0


def assert_exact_leg(y, ref):
    rel, mx, rms = errors(y, ref)
    assert rel <= EXACT_REL, f"rel-Frobenius {rel:.3e} > {EXACT_REL}"
    return rel
