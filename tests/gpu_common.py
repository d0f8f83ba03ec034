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


BF16_ULP = 2.0 ** -8   # spacing of bf16 values in [1, 2): a correctly rounded output is within half of it


def assert_close(name, got, want, tol):
    """Element-wise |got - want| <= tol, plus, for bf16 outputs (tol == BF16_TOL), the
    rounding of the output itself: one bf16 spacing relative to |want|. Without that
    term no bf16 output above 4 in magnitude could meet a 2e-2 absolute bound (its
    rounding alone can reach 2^-9 |x|)."""
    g = host(got) if hasattr(got, "detach") else np.asarray(got, dtype=np.float64)
    w = np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite output"
    if g.size == 0:
        return 0.0
    err = np.abs(g - w)
    bound = tol + (BF16_ULP * np.abs(w) if tol == BF16_TOL else 0.0)
    worst = int(np.argmax(err - bound))
    e, b = float(err.reshape(-1)[worst]), float(np.broadcast_to(bound, err.shape).reshape(-1)[worst])
    scale = float(np.abs(w).max())
    assert e <= b, (f"{name}: abs error {e:.3e} > bound {b:.3e} at |ref| {abs(float(w.reshape(-1)[worst])):.3g} "
                    f"(max abs error {float(err.max()):.3e}, max |ref| {scale:.3g})")
    return float(err.max())
