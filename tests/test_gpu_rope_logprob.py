"""GPU parity of depth-position RoPE and the shared-logit log-prob path."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, host, need_cuda, tma, torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,d,dtype", [("tiny_fp32", 64, "f32"), ("agentic_short", 128, "bf16"),
                                          ("galton_watson", 128, "bf16")])
def test_rope(name, d, dtype):
    need_cuda()
    m = tma()
    t = synth.CONFIGS[name]["tree"]()
    pk = m.tree_pack(t.seqs)
    ref = oracle.pack_ref(t.seqs)
    T = pk["T"]
    c = synth.CONFIGS[name]
    q, k, _, _ = synth.attention_config(name, T)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    tq, tk = dev(q, td), dev(k, td)
    pos = dev(pk["position_ids"])
    m.tree_rope(tq, tk, pos)
    tol = BF16_TOL if dtype == "bf16" else F32_TOL
    assert_close("rope q", tq, oracle.rope_ref(q, ref["paths"]), tol)
    assert_close("rope k", tk, oracle.rope_ref(k, ref["paths"]), tol)
    m.tree_rope(tq, tk, pos, inverse=True)
    assert_close("rope^-1 q", tq, q, 2 * tol)
    m.tree_check_device_status()


def _lm_case(T, K, V, n_occ_rows, bf16, seed, src=None):
    rng = np.random.default_rng(seed)
    if src is None:
        src = np.sort(rng.integers(0, n_occ_rows, size=3 * n_occ_rows)).astype(np.int32)
    h, w, tg, wt = synth.lm_head_config(T, K, V, len(src), bf16=bf16, seed=seed)
    order = np.argsort(src, kind="stable").astype(np.int32)
    row_ptr = np.zeros(T + 1, np.int32)
    row_ptr[1:] = np.cumsum(np.bincount(src, minlength=T))
    return h, w, src, tg, wt, row_ptr, order


def _run_lm(m, h, w, tg, wt, row_ptr, perm, bf16):
    td = torch.bfloat16 if bf16 else torch.float32
    th, tw = dev(h, td), dev(w, td)
    lse, logp = m.tree_logprob_fwd(th, tw, dev(row_ptr), dev(perm), dev(tg))
    g = (-wt).astype(np.float32)
    dh, dw = m.tree_logprob_bwd(th, tw, lse, dev(row_ptr), dev(perm), dev(tg), dev(g))
    m.tree_check_device_status()
    return lse, logp, dh, dw, g


@pytest.mark.parametrize("bf16", [True, False])
def test_logprob_without_occurrences(bf16):
    """Single-token sequences predict nothing: n_occ = 0. The forward still writes every
    row's LSE; the backward gives zero dH and dW."""
    need_cuda()
    m = tma()
    seqs = [[i] for i in range(150)]
    pk = m.tree_pack(seqs)
    assert pk["n_occ"] == 0
    T, K, V = pk["T"], 64, 520
    h, w, _, _ = synth.lm_head_config(T, K, V, 0, bf16=bf16)
    td = torch.bfloat16 if bf16 else torch.float32
    th, tw = dev(h, td), dev(w, td)
    empty = torch.zeros(0, dtype=torch.int32, device="cuda")
    lse, logp = m.tree_logprob_fwd(th, tw, dev(pk["occ_row_ptr"]), empty, empty)
    dh, dw = m.tree_logprob_bwd(th, tw, lse, dev(pk["occ_row_ptr"]), empty, empty,
                                torch.zeros(0, dtype=torch.float32, device="cuda"))
    m.tree_check_device_status()
    assert logp.numel() == 0
    z = h.astype(np.float64) @ w.astype(np.float64)
    zmax = z.max(axis=1, keepdims=True)
    want = (zmax + np.log(np.exp(z - zmax).sum(axis=1, keepdims=True)))[:, 0]
    assert_close("lse", lse, want, F32_TOL)
    assert float(dh.abs().max()) == 0.0 and float(dw.abs().max()) == 0.0


def test_logprob_tiny_fp32():
    need_cuda()
    m = tma()
    t = synth.tiny_tree()
    pk = m.tree_pack(t.seqs)
    h, w, _, _ = synth.lm_head_config(pk["T"], 64, 512, pk["n_occ"], bf16=False)
    wt = np.ones(pk["n_occ"], np.float32)
    lse, logp, dh, dw, g = _run_lm(m, h, w, pk["occ_targets"], wt, pk["occ_row_ptr"], pk["occ_perm"], False)
    rl, rlse = oracle.logprob_ref_fwd(h, w, pk["occ_source_rows"], pk["occ_targets"])
    used = np.unique(pk["occ_source_rows"])
    assert_close("logp", logp, rl, F32_TOL)
    assert_close("lse", host(lse)[used], rlse[used], F32_TOL)
    rdh, rdw = oracle.logprob_ref_bwd(h, w, pk["occ_source_rows"], pk["occ_targets"], g)
    assert_close("dH", dh, rdh, F32_TOL)
    assert_close("dW", dw, rdw, F32_TOL)


@pytest.mark.parametrize("T,K,V,bf16", [(200, 128, 1000, True), (333, 256, 4104, True), (130, 64, 520, False),
                                        (333, 128, 1000, False), (1500, 128, 4096, False)])
def test_logprob_random(T, K, V, bf16):
    """Ragged row/vocabulary tails, rows without occurrences, repeated targets; the last
    fp32 case has long contractions (dH over 4096 vocabulary columns, dW over 1500 rows)."""
    need_cuda()
    m = tma()
    h, w, src, tg, wt, row_ptr, perm = _lm_case(T, K, V, T - 7, bf16, seed=T)
    tg[::5] = tg[0]      # repeated targets across rows
    tg[1] = tg[2]        # and within a row
    lse, logp, dh, dw, g = _run_lm(m, h, w, tg, wt, row_ptr, perm, bf16)
    rl, rlse = oracle.logprob_ref_fwd(h, w, src, tg)
    used = np.unique(src)
    assert_close("logp", logp, rl, F32_TOL)
    assert_close("lse", host(lse)[used], rlse[used], F32_TOL)
    rdh, rdw = oracle.logprob_ref_bwd(h, w, src, tg, g)
    tol = BF16_TOL if bf16 else F32_TOL
    assert_close("dH", dh, rdh, tol)
    assert_close("dW", dw, rdw, tol)


def test_logprob_full_vocab_rows():
    """Full hidden and vocabulary sizes (4096 x 128256) on 256 rows: every output."""
    need_cuda()
    m = tma()
    T, K, V = 256, 4096, 128256
    h, w, src, tg, wt, row_ptr, perm = _lm_case(T, K, V, T, True, seed=7)
    lse, logp, dh, dw, g = _run_lm(m, h, w, tg, wt, row_ptr, perm, True)
    rl, rlse = oracle.logprob_ref_fwd(h, w, src, tg)
    assert_close("logp", logp, rl, F32_TOL)
    rdh, rdw = oracle.logprob_ref_bwd(h, w, src, tg, g)
    assert_close("dH", dh, rdh, BF16_TOL)
    assert_close("dW", dw, rdw, BF16_TOL)


def test_logprob_full_size_sampled():
    """The 8192-row tree at full size: sampled rows, and sum_v dW[k, v] = 0."""
    need_cuda()
    m = tma()
    t = synth.lm_head_tree()
    pk = m.tree_pack(t.seqs)
    T, K, V = pk["T"], 4096, 128256
    h, w, tg, wt = synth.lm_head_config(T, K, V, pk["n_occ"], bf16=True)
    lse, logp, dh, dw, g = _run_lm(m, h, w, tg, wt, pk["occ_row_ptr"], pk["occ_perm"], True)
    src = pk["occ_source_rows"]
    rng = np.random.default_rng(3)
    rows = rng.choice(np.unique(src), size=48, replace=False)
    sel = np.nonzero(np.isin(src, rows))[0]
    rl, rlse = oracle.logprob_ref_fwd(h, w, src[sel], tg[sel])
    assert_close("logp sampled", host(logp)[sel], rl, F32_TOL)
    assert_close("lse sampled", host(lse)[rows], rlse[rows], F32_TOL)
    gz = oracle.logprob_ref_gz(h, w, src, tg, g, rows)
    assert_close("dH sampled", host(dh)[rows], gz @ w.astype(np.float64).T, BF16_TOL)
    colsum = dw.float().sum(dim=1).double().cpu().numpy()
    assert np.abs(colsum).max() < 0.5, np.abs(colsum).max()


@pytest.mark.parametrize("T,K,V", [(200, 128, 1000), (333, 256, 4104)])
def test_logprob_dw_fp32(T, K, V):
    """dw_fp32: d_w written in fp32 straight from the accumulator. Its only rounding is
    that of the G_z operand the tensor cores read in bf16 (relative 2^-9 at cells other
    than the targets, whose exact values are added back), so per element
    |dW - ref| <= 1e-4 + 2^-8 sum_r |H[r, m]| |G_z[r, v]|, with G_z from the oracle."""
    need_cuda()
    m = tma()
    h, w, src, tg, wt, row_ptr, perm = _lm_case(T, K, V, T - 7, True, seed=T + 1)
    tg[::5] = tg[0]
    th, tw = dev(h, torch.bfloat16), dev(w, torch.bfloat16)
    lse, _ = m.tree_logprob_fwd(th, tw, dev(row_ptr), dev(perm), dev(tg))
    g = (-wt).astype(np.float32)
    dh, dw = m.tree_logprob_bwd(th, tw, lse, dev(row_ptr), dev(perm), dev(tg), dev(g), dw_fp32=True)
    m.tree_check_device_status()
    assert dw.dtype == torch.float32
    rdh, rdw = oracle.logprob_ref_bwd(h, w, src, tg, g)
    rows = np.arange(T)
    gz = oracle.logprob_ref_gz(h, w, src, tg, g, rows)
    bound = 1e-4 + 2.0 ** -8 * (np.abs(h.astype(np.float64)).T @ np.abs(gz))
    err = np.abs(dw.double().cpu().numpy() - rdw)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (float(err[worst]), float(bound[worst]), worst)
    assert_close("dH", dh, rdh, BF16_TOL)


def test_logprob_full_rows_and_vocab():
    """Every row of the 8192-row tree (18,475 occurrences over 8,174 rows, targets over the
    full 128,256-token vocabulary, some repeated) with hidden size 128: dH and dW, in bf16
    and in fp32, checked element-wise against one oracle pass everywhere, so the
    target-cell correction of dW runs at full occurrence density across every vocabulary
    block."""
    need_cuda()
    m = tma()
    t = synth.lm_head_tree()
    pk = m.tree_pack(t.seqs)
    T, K, V = pk["T"], 128, 128256
    h, w, tg, wt = synth.lm_head_config(T, K, V, pk["n_occ"], bf16=True)
    tg[::7] = tg[3]                     # a column that many occurrences share
    src = pk["occ_source_rows"]
    th, tw = dev(h, torch.bfloat16), dev(w, torch.bfloat16)
    row_ptr, perm = dev(pk["occ_row_ptr"]), dev(pk["occ_perm"])
    lse, logp = m.tree_logprob_fwd(th, tw, row_ptr, perm, dev(tg))
    g = (-wt).astype(np.float32)
    dh, dw = m.tree_logprob_bwd(th, tw, lse, row_ptr, perm, dev(tg), dev(g))
    _, dw32 = m.tree_logprob_bwd(th, tw, lse, row_ptr, perm, dev(tg), dev(g), dw_fp32=True)
    m.tree_check_device_status()
    rdh, rdw = oracle.logprob_ref_bwd(h, w, src, tg, g, chunk=512)
    assert_close("dH", dh, rdh, BF16_TOL)
    assert_close("dW (bf16)", dw, rdw, BF16_TOL)
    assert_close("dW (fp32)", dw32, rdw, BF16_TOL)
    # the fp32 output is the accumulator the bf16 output rounds
    assert torch.equal(dw32.to(torch.bfloat16), dw)
