"""Device-transfer helpers for the GPU parity tests (no method arithmetic)."""
import numpy as np


def dev(a):
    """numpy array -> torch CUDA tensor with the same bytes (uint16 -> int16)."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def bf16_dev(bits):
    import torch
    return dev(bits).view(torch.bfloat16)


def host(t):
    """torch tensor -> numpy float64 (bf16/fp16 widened exactly) or the integer dtype."""
    import torch
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32):
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def rms(a):
    return float(np.sqrt(np.mean(np.square(a))))


def gemm_error_ratio(y_gpu, y_ref, bf16_out):
    """max |err| / (1e-2 * RMS(ref) [+ bf16 half-ulp of ref]) -- <= 1 passes.

    The bound is 1e-2 * RMS of the oracle output; a bf16 output additionally
    carries its own rounding, at most 2^-8 * |y| (half a bf16 ulp)."""
    allowed = 1e-2 * rms(y_ref) + (2.0 ** -8 * np.abs(y_ref) if bf16_out else 0.0)
    return float(np.max(np.abs(y_gpu - y_ref) / allowed))
