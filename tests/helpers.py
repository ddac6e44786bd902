"""Shared helpers for the GPU parity tests: tolerance checks and host<->device marshalling."""
import numpy as np

MAX_ABS = 2e-2   # bf16 I/O, fp32 accumulation: max-abs bound on compressed KV and attention outputs
REL_L2 = 5e-3    # and relative L2 bound


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str, max_abs: float = MAX_ABS, rel_l2: float = REL_L2):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref).max() if got.size else 0.0
    den = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got - ref)
    assert err <= max_abs and rel <= rel_l2, f"{what}: max-abs {err:.3e} (<= {max_abs}), rel-L2 {rel:.3e} (<= {rel_l2})"
    return err, rel


def dev(a, torch, dtype=None):
    """numpy -> CUDA tensor keeping bit patterns (uint16 bf16 -> int16 storage)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.view(dtype)
