"""tree_attn_fwd_noalloc: the tree-attention forward for callers that cannot
allocate device memory for a workspace (for example when a framework's memory pool
already owns the device memory, or when a serving loop forbids cudaMalloc after
start-up). It keeps its scratch in a fixed array inside the library instead.

The tests call it through the C ABI, twice in a row each time, and check its output
against the float64 oracle and against tree_attn_fwd (which takes a caller
workspace) within the tolerances the other parity tests use: on a small tree on the
tensor-core path (bf16, d = 128) and on the fp32 path, and on a tree of exactly the
largest size the array serves (65,536 rows), where the last metadata tiles and the
padded subtree_end are in use. A tree larger than the array serves is refused with a
message. This file is collected last so that a failure here leaves the other tests
run."""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, need_cuda, tma, torch

pytestmark = pytest.mark.gpu

MAX_ROWS = 65536


def _noalloc(m, q, k, v, end, o, lse, dtype_code):
    T, Hq, d = q.shape
    rc = m.lib().tree_attn_fwd_noalloc(
        C.c_void_p(q.data_ptr()), C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()),
        C.c_void_p(o.data_ptr()), C.c_void_p(lse.data_ptr()), C.c_void_p(end.data_ptr()),
        T, Hq, k.shape[1], d, dtype_code, 0.0, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


def _call_twice(m, q, k, v, end, bf):
    """Two calls in a row into fresh NaN-filled outputs; returns both results."""
    T, Hq, _ = q.shape
    res = []
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((Hq, T), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(m, q, k, v, end, o, lse, 1 if bf else 0) == 0, m.lib().tree_last_error()
        m.tree_check_device_status()
        res.append((o, lse))
    return res


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_noalloc_forward_matches_oracle_and_workspace_forward(dtype, d):
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=6, budget=900, seg=(10, 150), vocab=1000)
    pk = m.tree_pack(t.seqs)
    ref = oracle.pack_ref(t.seqs)
    T = pk["T"]
    bf = dtype == "bf16"
    td = torch.bfloat16 if bf else torch.float32
    qh, kh, vh = (synth.normal(s, shape, bf16=bf) for s, shape in ((61, (T, 4, d)), (62, (T, 2, d)), (63, (T, 2, d))))
    q, k, v = dev(qh, td), dev(kh, td), dev(vh, td)
    end = dev(pk["subtree_end"])
    want_o, want_lse = oracle.attn_ref_fwd(qh, kh, vh, ref["paths"])
    o_ws, lse_ws = m.tree_attn_fwd(q, k, v, end)
    tol = BF16_TOL if bf else F32_TOL
    for o, lse in _call_twice(m, q, k, v, end, bf):
        assert_close("O (no-alloc vs oracle)", o, want_o, tol)
        assert_close("LSE (no-alloc vs oracle)", lse, want_lse, F32_TOL)
        assert_close("O (no-alloc vs workspace)", o, o_ws.double().cpu().numpy(), tol)
        assert_close("LSE (no-alloc vs workspace)", lse, lse_ws.double().cpu().numpy(), F32_TOL)


def test_noalloc_forward_at_its_largest_tree():
    """T = 65,536 exactly (a Galton-Watson tree clipped to that budget), bf16, d = 128:
    every row against tree_attn_fwd with a workspace (the same kernel: bitwise equal),
    and rows sampled across the whole tree -- the last two 128-row tiles included --
    against the oracle."""
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=3, budget=MAX_ROWS, max_depth=9, seg=(64, 512), vocab=32000)
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    assert T == MAX_ROWS
    qh, kh, vh = (synth.normal(s, shape, bf16=True) for s, shape in
                  ((71, (T, 2, 128)), (72, (T, 1, 128)), (73, (T, 1, 128))))
    q, k, v = (dev(x, torch.bfloat16) for x in (qh, kh, vh))
    end = dev(pk["subtree_end"])
    o_ws, lse_ws = m.tree_attn_fwd(q, k, v, end)
    r = np.random.default_rng(5)
    rows = np.unique(np.concatenate([r.choice(T, 160, replace=False), np.arange(T - 256, T, 7), [0, T - 1]]))
    ref = oracle.pack_ref(t.seqs)
    want_o, want_lse = oracle.attn_ref_rows(qh, kh, vh, ref["paths"], rows)
    for o, lse in _call_twice(m, q, k, v, end, True):
        assert torch.equal(o, o_ws), "no-alloc forward differs from the workspace forward"
        assert torch.equal(lse, lse_ws), "no-alloc LSE differs from the workspace forward"
        assert_close("O rows (no-alloc vs oracle)", o[torch.from_numpy(rows).cuda()], want_o, BF16_TOL)
        assert_close("LSE rows (no-alloc vs oracle)", lse[:, torch.from_numpy(rows).cuda()], want_lse, F32_TOL)


def test_noalloc_refuses_trees_beyond_its_scratch():
    need_cuda()
    m = tma()
    T = MAX_ROWS + 128
    q = torch.zeros((T, 2, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((T, 1, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, T), dtype=torch.float32, device="cuda")
    end = torch.arange(T, dtype=torch.int32, device="cuda")
    assert _noalloc(m, q, k, k, end, q, lse, 1) == 2
    assert b"65536" in m.lib().tree_last_error()
