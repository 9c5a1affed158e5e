"""Shared helpers of the GPU parity tests (no arithmetic of the layer here)."""
import numpy as np
import torch

# Acceptance bound on bf16 outputs: max |gpu - oracle| <= 2e-2 * max |oracle|.
OUT_RTOL = 2e-2
# Router weights: fp32 expf/division on the GPU vs fp64 in the oracle.
W_RTOL = 1e-5
W_ATOL = 1e-7


def rel_max_err(got: np.ndarray, ref: np.ndarray) -> float:
    scale = np.abs(ref).max()
    return float(np.abs(got - ref).max() / scale) if scale > 0 else float(np.abs(got).max())


def assert_out_close(out_gpu: torch.Tensor, ref: np.ndarray, rows=None, tol=OUT_RTOL):
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    assert np.all(np.isfinite(got))
    err = rel_max_err(got, ref)
    assert err <= tol, f"max|gpu-oracle| / max|oracle| = {err:.3e} > {tol}"
    return err


def sample_rows(T: int, n: int, seed: int = 0):
    """All rows when T <= n, else first, last and random rows (sorted)."""
    if T <= n:
        return list(range(T))
    rng = np.random.default_rng(seed)
    pick = set([0, T - 1]) | set(rng.choice(T, n - 2, replace=False).tolist())
    return sorted(pick)
