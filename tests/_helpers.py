"""Shared test helpers: tolerances and tensor <-> oracle conversion."""

import numpy as np
import torch

# Attention outputs against the fp64 oracle (bf16 inputs, fp32 accumulation,
# bf16 output): max-abs <= 1e-2 and relative L2 <= 5e-3.
MAX_ABS = 1e-2
REL_L2 = 5e-3


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a (bf16) tensor, on the CPU."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_attn_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = np.abs(got - want)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(got - want) / denom) if denom > 0 else float(np.linalg.norm(got - want))
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def bits(t: torch.Tensor) -> torch.Tensor:
    """Raw 16-bit patterns of a bf16 tensor (for bit-exact comparisons)."""
    return t.contiguous().view(torch.int16)
