"""Comparison helpers for the GPU parity tests (test infrastructure)."""
import numpy as np

# Tolerances of the target: bf16 inputs (fp32 accumulation and outputs):
# max-abs <= 2e-2 and relative L2 <= 1e-2; fp32 inputs: relative L2 <= 1e-4.
BF16_MAX_ABS, BF16_REL_L2, F32_REL_L2 = 2e-2, 1e-2, 1e-4
# Secondary criterion printed by the pages for bf16 kernels: |d| <= atol + rtol |ref|.
PAGE_ATOL, PAGE_RTOL = 1e-2, 1e-2


def stats(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = np.abs(got - ref)
    rel = float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))
    return dict(max_abs=float(d.max()) if d.size else 0.0, rel_l2=rel,
                diff_mean=float(d.mean()) if d.size else 0.0,
                page_ok=bool(np.all(d <= PAGE_ATOL + PAGE_RTOL * np.abs(ref))))


def assert_close(name, got, ref, dtype):
    s = stats(got, ref)
    if dtype == "f32":
        ok = s["rel_l2"] <= F32_REL_L2
    else:
        ok = s["max_abs"] <= BF16_MAX_ABS and s["rel_l2"] <= BF16_REL_L2
    assert ok, f"{name}: {s}"
    return s


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
