"""Helpers shared by the GPU parity tests: moving the seeded inputs to the
device bit-for-bit and the error measures the tolerances are stated in."""
import numpy as np
import torch


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy input (bf16 bit patterns as uint16, or float32) -> torch CUDA tensor, same bits."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


# tolerances (fp32: max-abs on O, dQ, dK, dV; bf16: O max-abs, gradients relative L2)
FP32_MAX_ABS = 1e-5
BF16_O_MAX_ABS = 2e-2
BF16_GRAD_REL_L2 = 1e-2
STAT_REL = 1e-3   # m and l (informative bound)


def check_stats(m, l, om, ol):
    m, l = host(m), host(l)
    fin = np.isfinite(om)
    assert np.array_equal(np.isfinite(m), fin), "rows with no allowed key disagree"
    if fin.any():
        assert np.max(np.abs(m[fin] - om[fin]) / (1 + np.abs(om[fin]))) <= STAT_REL
        assert np.max(np.abs(l[fin] - ol[fin]) / np.abs(ol[fin])) <= STAT_REL
    assert np.all(l[~fin] == 0)
