"""Helpers of the GPU parity tests: host <-> device transfers of exact bit patterns
and the comparison rules. Holds none of the block's arithmetic."""
import numpy as np
import pytest

try:
    import torch
except ImportError:  # pragma: no cover
    torch = None


def need_gpu():
    if torch is None or not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def dev_bf16(bits: np.ndarray):
    """uint16 bf16 bit patterns -> CUDA bfloat16 tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f64(t) -> np.ndarray:
    """Exact float64 copy of a CUDA float32 / bfloat16 tensor."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return t.contiguous().cpu().numpy().astype(np.float64)


def host_bits_f32(t) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint32)


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max|got - ref| / max|ref| (the normalised bound used by every fp test)."""
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref))) / scale


BF16_TOL = 1e-2   # bf16 inputs, fp32 accumulation: max|Y_gpu - Y_ref| <= 1e-2 * max|Y_ref|
F32_TOL = 1e-5    # fp32 inputs, fp32 FMA accumulation


def assert_close(got, ref, tol, what=""):
    err = max_rel_err(got, ref)
    assert err <= tol, f"{what}: normalised error {err:.3e} > {tol:.0e}"
    return err
