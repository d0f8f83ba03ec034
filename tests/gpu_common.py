"""Helpers for the GPU parity tests: device tensors from the seeded generators,
oracle inputs from the same (bf16-rounded) values, error reporting."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

BF16_TOL = 2e-2     # max abs error of bf16 outputs against the float64 oracle
F32_TOL = 1e-4      # max abs error of fp32 outputs (LSE, logp; every output of an fp32 run)


def need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def tma():
    import __graft_entry__
    __graft_entry__.build()
    import tree_masked_attention_gb300 as m
    return m


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(dtype) if dtype is not None else t


def host(t):
    return t.detach().double().cpu().numpy()


def max_err(got, want):
    got = host(got) if hasattr(got, "detach") else np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), "non-finite output"
    return float(np.abs(got - want).max()) if got.size else 0.0


def assert_close(name, got, want, tol):
    e = max_err(got, want)
    scale = float(np.abs(np.asarray(want, dtype=np.float64)).max()) if np.size(want) else 0.0
    assert e <= tol, f"{name}: max abs error {e:.3e} > {tol:.1e} (max |ref| {scale:.3g})"
    return e
