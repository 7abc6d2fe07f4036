"""Helpers shared by the tests: tensor <-> bf16-bit conversions and the
output tolerances.

Tolerance on outputs y (and on the activation a): with y_ref the oracle's
values, max|y - y_ref| <= 2e-2 * max|y_ref| and the relative L1 error
sum|y - y_ref| / sum|y_ref| <= 5e-3.  Routing outputs are compared bit for
bit; router weights to 1e-6 absolute.
"""
import numpy as np
import torch

Y_MAX_REL = 2e-2
Y_MEAN_REL = 5e-3
W_ABS = 1e-6


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64_of_bits(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tensor_of_bits(b, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def assert_close_bf16(got_bits, ref_bits, what="y", max_rel=Y_MAX_REL, mean_rel=Y_MEAN_REL):
    g = f64_of_bits(got_bits)
    r = f64_of_bits(ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - r)
    scale = np.abs(r).max()
    l1 = np.abs(r).sum()
    if scale == 0:
        assert err.max() == 0, f"{what}: expected zeros"
        return
    assert err.max() <= max_rel * scale, f"{what}: max|err| {err.max():.4e} > {max_rel} * {scale:.4e}"
    assert err.sum() <= mean_rel * l1, f"{what}: rel L1 {err.sum() / l1:.4e} > {mean_rel}"


def fp32_dot_error_bound(x_f64, w_f64):
    """Bound on |fp32 dot - exact| for each entry of x @ w.T: K * 2^-24 * sum|x w|
    (the standard bound for any fp32 summation order of K products; each
    product of two bf16 values is exact in fp32)."""
    K = x_f64.shape[1]
    return K * 2.0 ** -24 * (np.abs(x_f64) @ np.abs(w_f64).T)
