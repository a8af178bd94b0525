"""Comparison helpers for the parity tests (GPU result vs CPU oracle)."""
import numpy as np
import torch

# Tolerances, as |C - C_ref| <= REL * absAB + ABS, with absAB = sum_k |A||B|.
F32_REL, F32_ABS = 1e-5, 1e-6      # FP32 CUDA-core path
TC_REL, TC_ABS = 1e-2, 0.0         # TF32 / BF16 tensor-core path


def to_np(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def assert_within(C, C_ref, absAB, rel, abs_, what=""):
    C = to_np(C)
    assert C.shape == C_ref.shape, (C.shape, C_ref.shape)
    assert np.isfinite(C).all(), f"{what}: non-finite output"
    err = np.abs(C - C_ref)
    bound = rel * absAB + abs_
    bad = err > bound
    if bad.any():
        i, j = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs out of tolerance; worst at "
            f"({i},{j}): got {C[i, j]!r}, oracle {C_ref[i, j]!r}, bound {bound[i, j]:.3e}")
    return float((err / np.maximum(absAB, 1e-30)).max()) if err.size else 0.0


def assert_bit_exact(C, C_ref, what=""):
    C = to_np(C)
    ref32 = C_ref.astype(np.float32).astype(np.float64)
    assert np.array_equal(ref32, C_ref), f"{what}: oracle value not representable in fp32"
    if not np.array_equal(C, C_ref):
        diff = np.argwhere(C != C_ref)
        i, j = diff[0]
        raise AssertionError(f"{what}: {len(diff)} outputs differ; first at ({i},{j}): "
                             f"got {C[i, j]!r}, oracle {C_ref[i, j]!r}")
