"""Helpers for the GPU parity tests: device copies of synthetic inputs and the
comparison metrics (max-abs, cosine) the tolerances are stated in."""
import numpy as np
import torch


def dev_f16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float16))).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.float().cpu().numpy().astype(np.float64)


def decode_e4m3(codes: torch.Tensor) -> np.ndarray:
    """E4M3 codes of 16*x -> x (torch's float8_e4m3fn view is the library decoder)."""
    return codes.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy() / 16.0


def cosine_rows(a, b) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64).reshape(len(a), -1)
    b = np.asarray(b, dtype=np.float64).reshape(len(b), -1)
    return (a * b).sum(1) / (np.linalg.norm(a, axis=1) * np.linalg.norm(b, axis=1))


def assert_close(got, ref, rtol, atol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} elements out of tolerance; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} (max abs err {err.max():.3e})")
