"""GPU parity of tree attention (forward and backward) against the oracle."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, host, need_cuda, tma, torch

pytestmark = pytest.mark.gpu


def _run(m, pk, q, k, v, do, dtype, deterministic=False):
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    tq, tk, tv, tdo = (dev(x, td) for x in (q, k, v, do))
    end = dev(pk["subtree_end"])
    o, lse = m.tree_attn_fwd(tq, tk, tv, end)
    dq, dk, dv = m.tree_attn_bwd(tq, tk, tv, o, tdo, lse, end, deterministic=deterministic)
    m.tree_check_device_status()
    return o, lse, dq, dk, dv


def _full_check(seqs, Hq, Hkv, d, dtype, seed=0, deterministic=False):
    need_cuda()
    m = tma()
    pk = m.tree_pack(seqs)
    T = pk["T"]
    bf = dtype == "bf16"
    q = synth.normal(10 * seed + 1, (T, Hq, d), bf16=bf)
    k = synth.normal(10 * seed + 2, (T, Hkv, d), bf16=bf)
    v = synth.normal(10 * seed + 3, (T, Hkv, d), bf16=bf)
    do = synth.normal(10 * seed + 4, (T, Hq, d), bf16=bf)
    o, lse, dq, dk, dv = _run(m, pk, q, k, v, do, dtype, deterministic)
    ref = oracle.pack_ref(seqs)
    ro, rlse = oracle.attn_ref_fwd(q, k, v, ref["paths"])
    rdq, rdk, rdv = oracle.attn_ref_bwd(q, k, v, do, ref["paths"])
    tol = BF16_TOL if bf else F32_TOL
    assert_close("O", o, ro, tol)
    assert_close("LSE", lse, rlse, F32_TOL)
    assert_close("dQ", dq, rdq, tol)
    assert_close("dK", dk, rdk, tol)
    assert_close("dV", dv, rdv, tol)
    return m, pk, (q, k, v, do), (o, lse, dq, dk, dv)


def test_tiny_tree_fp32():
    t = synth.tiny_tree()
    _full_check(t.seqs, 1, 1, 64, "f32")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_trees(d, dtype, seed):
    """Galton-Watson trees of a few hundred rows: several 128-row tiles and a ragged tail."""
    t = synth.galton_watson(seed=seed, budget=[333, 517, 700][seed], seg=(5, 90), vocab=1000)
    _full_check(t.seqs, 4, 2, d, dtype, seed=seed)


def test_fp32_head64_deeper_tree():
    """fp32 at head size 64 (the tf32-split kernels) on a Galton-Watson tree of about 3000
    rows: paths up to ~1500 rows, so dQ sums over dozens of key tiles and dK/dV over many
    query tiles, every partial added in fp32 outside the tensor cores."""
    t = synth.galton_watson(seed=21, budget=3000, seg=(40, 300), vocab=1000)
    _full_check(t.seqs, 4, 2, 64, "f32", seed=21)


@pytest.mark.parametrize("Hq,Hkv", [(3, 1), (8, 8), (8, 2), (6, 3)])
def test_group_sizes(Hq, Hkv):
    """Odd and even GQA groups, MHA: the tensor-core kernels and their fallbacks."""
    t = synth.galton_watson(seed=9, budget=600, seg=(5, 90), vocab=1000)
    _full_check(t.seqs, Hq, Hkv, 128, "bf16", seed=9)


def test_deterministic_matches_default():
    """Both backward modes agree with the oracle (and so with each other)."""
    t = synth.galton_watson(seed=8, budget=640, seg=(5, 90), vocab=1000)
    _full_check(t.seqs, 4, 2, 128, "bf16", seed=8, deterministic=True)


def test_deterministic_short_prompt_agentic_full_size():
    """The deterministic backward (one work unit per key tile for dK / dV, query-stationary
    dQ in key-tile order) on the full short-prompt agentic tree, against the oracle."""
    t = synth.agentic_short()
    _full_check(t.seqs, 32, 8, 128, "bf16", seed=5, deterministic=True)


def test_short_prompt_agentic_full_size():
    """The short-prompt agentic tree at full size (T = 2304, 32/8 heads, d = 128, bf16)."""
    t = synth.agentic_short()
    _full_check(t.seqs, 32, 8, 128, "bf16")


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("case", ["chain", "forest_of_singletons", "single_token", "two_roots"])
def test_degenerate_trees(case, dtype, d):
    rng = np.random.default_rng(5)
    if case == "chain":
        seqs = [rng.integers(0, 100, size=1000)]
    elif case == "forest_of_singletons":
        seqs = [[i] for i in range(300)]
    elif case == "single_token":
        seqs = [[42]]
    else:
        seqs = [rng.integers(0, 100, size=200), [1000] + list(rng.integers(0, 100, size=150))]
    _full_check(seqs, 2, 1, d, dtype)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_deterministic_flag_repeats_bitwise(dtype, d):
    """bf16 at d = 128 on the kind::f16 kernels; fp32 and bf16 at d = 64 on the tf32-split
    kernels (whose backward has one fixed summation order whatever the flag)."""
    need_cuda()
    t = synth.galton_watson(seed=4, budget=600, seg=(5, 90), vocab=1000)
    m = tma()
    pk = m.tree_pack(t.seqs)
    if d == 128:
        q, k, v, do = synth.attention_config("agentic_short", pk["T"], seed=3)
    else:
        T, bf = pk["T"], dtype == "bf16"
        q, k, v, do = (synth.normal(30 + s, shape, bf16=bf) for s, shape in
                       enumerate(((T, 8, d), (T, 2, d), (T, 2, d), (T, 8, d))))
    r1 = _run(m, pk, q, k, v, do, dtype, deterministic=True)
    r2 = _run(m, pk, q, k, v, do, dtype, deterministic=True)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)
    if d == 64:
        r3 = _run(m, pk, q, k, v, do, dtype, deterministic=False)
        for a, b in zip(r1, r3):
            assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["agentic_long", "galton_watson"])
def test_full_size_sampled(name):
    """T = 16k workloads: sampled rows against the oracle row by row, plus the
    identities sum_j dV_j = sum_i dO_i (per KV group) and sum_j dK_j = 0."""
    need_cuda()
    m = tma()
    t = synth.CONFIGS[name]["tree"]()
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    q, k, v, do = synth.attention_config(name, T)
    o, lse, dq, dk, dv = _run(m, pk, q, k, v, do, "bf16")
    ref = oracle.pack_ref(t.seqs)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([[0, 1, T - 1], rng.integers(0, T, size=24)]))
    ro, rlse = oracle.attn_ref_rows(q, k, v, ref["paths"], rows)
    assert_close("O rows", host(o)[rows], ro, BF16_TOL)
    assert_close("LSE rows", host(lse)[:, rows], rlse, F32_TOL)
    assert_close("dQ rows", host(dq)[rows], oracle.attn_ref_dq_rows(q, k, v, do, ref["paths"], rows), BF16_TOL)
    # keys with small subtrees (cheap to sum over every descendant query)
    size = pk["subtree_end"] - np.arange(T) + 1
    small = np.nonzero(size <= 300)[0]
    keys = np.unique(np.concatenate([[T - 1], rng.choice(small, size=12, replace=False)]))
    rdk, rdv = oracle.attn_ref_dkdv_rows(q, k, v, do, ref["paths"], keys)
    assert_close("dK rows", host(dk)[keys], rdk, BF16_TOL)
    assert_close("dV rows", host(dv)[keys], rdv, BF16_TOL)
    g = q.shape[1] // k.shape[1]
    sum_do = do.astype(np.float64).reshape(T, k.shape[1], g, -1).sum(axis=(0, 2))
    assert_close("sum dV", host(dv).sum(0), sum_do, 0.5)
    assert_close("sum dK", host(dk).sum(0), np.zeros_like(sum_do), 0.5)


@pytest.mark.parametrize("name,g", [("agentic_long", 5), ("galton_watson", 2)])
def test_full_size_one_kv_group_every_row(name, g):
    """The 16k-row trees at full size (32 / 8 heads): every row of O, LSE and dQ of the four
    query heads of KV group g, and every row of that group's dK and dV -- the prompt and
    root keys, whose subtrees hold every query, included -- against the per-path oracle
    run on that group alone (KV groups are independent, so the group's slice of the inputs
    is a complete problem of its own)."""
    need_cuda()
    m = tma()
    t = synth.CONFIGS[name]["tree"]()
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    q, k, v, do = synth.attention_config(name, T)
    o, lse, dq, dk, dv = _run(m, pk, q, k, v, do, "bf16")
    G = q.shape[1] // k.shape[1]
    hs = slice(G * g, G * (g + 1))
    paths = oracle.pack_ref(t.seqs)["paths"]
    sq, sk, sv, sdo = q[:, hs], k[:, g:g + 1], v[:, g:g + 1], do[:, hs]
    ro, rlse = oracle.attn_ref_fwd(sq, sk, sv, paths)
    rdq, rdk, rdv = oracle.attn_ref_bwd(sq, sk, sv, sdo, paths)
    assert_close("O", host(o)[:, hs], ro, BF16_TOL)
    assert_close("LSE", host(lse)[hs], rlse, F32_TOL)
    assert_close("dQ", host(dq)[:, hs], rdq, BF16_TOL)
    assert_close("dK", host(dk)[:, g:g + 1], rdk, BF16_TOL)
    assert_close("dV", host(dv)[:, g:g + 1], rdv, BF16_TOL)


def test_bad_subtree_end_sets_device_flag():
    """An out-of-range subtree_end is reported through the device error word;
    the kernels never index memory with it, so nothing faults."""
    need_cuda()
    m = tma()
    T = 200
    end = np.arange(T, dtype=np.int32)
    end[17] = T + 5
    q = torch.zeros((T, 2, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((T, 1, 64), dtype=torch.bfloat16, device="cuda")
    m.tree_attn_fwd(q, k, k, dev(end))
    with pytest.raises(m.TreeError) as ei:
        m.tree_check_device_status()
    assert ei.value.status == 7
    m.tree_check_device_status()   # cleared


def test_kernel_timing_brackets():
    """tree_kernel_timing brackets the main kernels; durations come back positive."""
    need_cuda()
    m = tma()
    t = synth.galton_watson(seed=3, budget=400, seg=(5, 90), vocab=1000)
    pk = m.tree_pack(t.seqs)
    T = pk["T"]
    q, k, v, do = (dev(synth.normal(s, (T, h, 128), bf16=True), torch.bfloat16)
                   for s, h in ((1, 4), (2, 2), (3, 2), (4, 4)))
    end = dev(pk["subtree_end"])
    m.tree_kernel_timing(True)
    try:
        o, lse = m.tree_attn_fwd(q, k, v, end)
        m.tree_attn_bwd(q, k, v, o, do, lse, end)
        assert m.tree_kernel_last_ms(0) > 0 and m.tree_kernel_last_ms(1) > 0
        assert m.tree_kernel_last_ms(2) == -1
    finally:
        m.tree_kernel_timing(False)
    m.tree_check_device_status()


def test_fma_exp2_matches_hardware_exp2():
    """The FMA-pipe 2^x used for part of the forward softmax's exponentials: relative error
    within 1e-5 of CUDA's exp2 over the softmax's range, exact powers of two at integers,
    and 2^-125 below -125 (where the SFU's ftz ex2 gives 0 or a denormal)."""
    need_cuda()
    m = tma()
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-125.0, 0.0, 200000), rng.uniform(-2.0, 2.0, 50000),
                        np.arange(-125, 21, dtype=np.float64), np.arange(-125, 20) + 0.5,
                        [-0.5, 0.5, -1e-7, 1e-7, 0.0]]).astype(np.float32)
    tx = torch.from_numpy(x).cuda()
    y = m.tree_selftest_exp2(tx)
    ref = torch.exp2(tx.double())
    rel = ((y.double() - ref).abs() / ref).cpu().numpy()
    assert rel.max() <= 1e-5, float(rel.max())
    ints = np.arange(-125, 21)
    yi = m.tree_selftest_exp2(torch.from_numpy(ints.astype(np.float32)).cuda()).cpu().numpy()
    assert np.allclose(yi, 2.0 ** ints, rtol=3e-6, atol=0)
    low = m.tree_selftest_exp2(torch.tensor([-126.0, -200.0, -float("inf")], device="cuda")).cpu().numpy()
    assert np.allclose(low, 2.0 ** -125, rtol=1e-5, atol=0)
