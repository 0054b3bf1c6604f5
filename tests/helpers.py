"""Shared helpers of the GPU tests: device transfer and the error metrics.

Tolerances (the contract of the path):
  * fp32 I/O: max |out - ref| <= 1e-5 over all elements;
  * bf16 I/O: for every row i, max_d |out - ref| / max_d |ref_i| <= 4e-3
    ("relative to the row max-norm"; A and Z_k are fp32 inside);
  * graphs: bit-exact CSR.
"""
import numpy as np

FP32_ABS_TOL = 1e-5
BF16_ROW_TOL = 4e-3


def to_device(x: np.ndarray, dtype: str, device="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(device)


def to_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def row_relative_error(got: np.ndarray, ref: np.ndarray) -> float:
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    den = np.where(den > 0, den, 1.0)
    return float((num / den).max()) if num.size else 0.0


def check_output(got: np.ndarray, ref: np.ndarray, dtype: str) -> float:
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    if dtype == "fp32":
        err = float(np.abs(got - ref).max()) if got.size else 0.0
        assert err <= FP32_ABS_TOL, f"fp32 max-abs error {err:.3e} > {FP32_ABS_TOL}"
    else:
        err = row_relative_error(got, ref)
        assert err <= BF16_ROW_TOL, f"bf16 row-relative error {err:.3e} > {BF16_ROW_TOL}"
    return err
