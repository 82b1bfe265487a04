"""Shared helpers of the GPU parity tests: put global-order inputs into the
sharded order with the ORACLE's shard map (so attention tests do not depend on
the GPU permutation kernel), run the library, bring results back to global
order, and the error measures the tolerances are stated in."""

import numpy as np
import torch

import oracle

BF16_O_ATOL = 2e-2     # max abs on o
BF16_LSE_ATOL = 1e-3   # max abs on lse
BF16_GRAD_RFRO = 2e-2  # relative Frobenius on dq, dk, dv
F32_ATOL = 1e-5        # max abs, fp32 runs


def perm_of(cu, C, layout):
    return torch.from_numpy(oracle.shard_order(cu, C, layout))


def to_dev_sharded(x: torch.Tensor, perm: torch.Tensor) -> torch.Tensor:
    return x.index_select(0, perm).contiguous().cuda()


def to_host_global(xs: torch.Tensor, perm: torch.Tensor) -> torch.Tensor:
    xs = xs.cpu()
    out = torch.empty_like(xs)
    out[perm] = xs
    return out


def lse_to_global(lse_s: torch.Tensor, perm: torch.Tensor) -> torch.Tensor:
    lse_s = lse_s.cpu()
    out = torch.empty_like(lse_s)
    out[:, perm] = lse_s
    return out


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / max(den, 1e-30))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()
