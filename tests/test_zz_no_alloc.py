"""tree_attn_fwd_noalloc: the tree-attention forward for callers that cannot
allocate device memory for a workspace (for example when a framework's memory pool
already owns the device memory, or when a serving loop forbids cudaMalloc after
start-up). It keeps its scratch in a fixed array inside the library instead.

The test calls it through the C ABI and checks, on two calls in a row, that its
output matches tree_attn_fwd (which takes a caller workspace) within the tolerance
the other parity tests use, on the tensor-core path (bf16, d = 128) and on the
fp32 path; and that a tree larger than the array serves is refused with a message.
This file is collected last so that a failure here leaves the other tests run."""
import ctypes as C

import numpy as np
import pytest

import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, need_cuda, tma, torch

pytestmark = pytest.mark.gpu


def _noalloc(m, q, k, v, end, o, lse, dtype_code):
    T, Hq, d = q.shape
    rc = m.lib().tree_attn_fwd_noalloc(
        C.c_void_p(q.data_ptr()), C.c_void_p(k.data_ptr()), C.c_void_p(v.data_ptr()),
        C.c_void_p(o.data_ptr()), C.c_void_p(lse.data_ptr()), C.c_void_p(end.data_ptr()),
        T, Hq, k.shape[1], d, dtype_code, 0.0, C.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_noalloc_forward_matches_workspace_forward(dtype, d):
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=6, budget=900, seg=(10, 150), vocab=1000)
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    bf = dtype == "bf16"
    td = torch.bfloat16 if bf else torch.float32
    q = dev(synth.normal(61, (T, 4, d), bf16=bf), td)
    k = dev(synth.normal(62, (T, 2, d), bf16=bf), td)
    v = dev(synth.normal(63, (T, 2, d), bf16=bf), td)
    end = dev(pk["subtree_end"])
    o_ref, lse_ref = m.tree_attn_fwd(q, k, v, end)
    tol = BF16_TOL if bf else F32_TOL
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((4, T), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(m, q, k, v, end, o, lse, 1 if bf else 0) == 0, m.lib().tree_last_error()
        m.tree_check_device_status()
        assert_close("O (no-alloc vs workspace)", o, o_ref.double().cpu().numpy(), tol)
        assert_close("LSE (no-alloc vs workspace)", lse, lse_ref.double().cpu().numpy(), F32_TOL)


def test_noalloc_refuses_trees_beyond_its_scratch():
    need_cuda()
    m = tma()
    T = 65536 + 128
    q = torch.zeros((T, 2, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((T, 1, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, T), dtype=torch.float32, device="cuda")
    end = torch.arange(T, dtype=torch.int32, device="cuda")
    assert _noalloc(m, q, k, k, end, q, lse, 1) == 2
    assert b"65536" in m.lib().tree_last_error()
