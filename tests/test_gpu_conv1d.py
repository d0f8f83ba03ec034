"""GPU parity of the tree-correct causal depthwise conv1d (Tree Training §3.2 "(ii)
Causal convolution", eq. 11, Fig. 4) with the per-branch oracle: forward y, backward
dx, dw, dbias, on random forests, the tiny tree and the 16384-row Galton-Watson tree."""
import numpy as np
import pytest

import oracle
import synth
from gpu_common import BF16_TOL, F32_TOL, assert_close, dev, host, need_cuda, tma, torch

pytestmark = pytest.mark.gpu


def _run(m, seqs, C, K, bf16, seed, bias=True, channels=None):
    """GPU forward + backward on the packed tree; oracle on `channels` (all by default)."""
    pk = m.tree_pack(seqs)
    ref = oracle.pack_ref(seqs)
    T = pk["T"]
    x, w, b, dy = synth.conv1d_config(T, C, K, bf16, seed)
    td = torch.bfloat16 if bf16 else torch.float32
    tx, tw, tdy = dev(x, td), dev(w, td), dev(dy, td)
    tb = dev(b, td) if bias else None
    y = m.tree_conv1d_fwd(tx, tw, dev(pk["parent_row"]), bias=tb)
    dx, dw, db = m.tree_conv1d_bwd(tx, tw, tdy, dev(pk["subtree_end"]), dev(pk["position_ids"]))
    m.tree_check_device_status()
    cs = np.arange(C) if channels is None else np.asarray(channels)
    tcs = torch.from_numpy(cs).cuda()
    xs, ws_, dys = x[:, cs], w[cs], dy[:, cs]
    bs = b[cs] if bias else None
    ry = oracle.conv1d_ref_fwd(xs, ws_, ref["paths"], bs)
    rdx, rdw, rdb = oracle.conv1d_ref_bwd(xs, ws_, dys, ref["paths"], bs)
    tol = BF16_TOL if bf16 else F32_TOL
    assert_close("y", y[:, tcs], ry, tol)
    assert_close("dx", dx[:, tcs], rdx, tol)
    # dw and dbias are sums over all T rows: fp32 sums of 64 rows per tile, then fp64
    # over tiles, so their rounding is at most (64 + 2) * 2^-24 * (sum of |terms|); the
    # sum of |terms| is the same gradient taken on |x| and |dy|
    _, adw, adb = oracle.conv1d_ref_bwd(np.abs(xs), ws_, np.abs(dys), ref["paths"])
    u = 66 * 2.0 ** -24
    gdw, gdb = host(dw[tcs]), host(db[tcs])
    assert np.all(np.abs(gdw - rdw) <= F32_TOL + u * adw), float(np.abs(gdw - rdw).max())
    assert np.all(np.abs(gdb - rdb) <= F32_TOL + u * adb), float(np.abs(gdb - rdb).max())
    return pk


@pytest.mark.parametrize("seed,C,K,bf16", [(0, 8, 1, False), (1, 64, 2, False), (2, 64, 3, True),
                                           (3, 520, 4, True), (4, 128, 4, False), (5, 72, 8, True),
                                           (6, 16, 5, False)])
def test_conv1d_random_forests(seed, C, K, bf16):
    """Random forests of short sequences over a small vocabulary (many forks, several
    roots), T ragged against the 32/64-row tiles; C = 520 spans two channel tiles."""
    need_cuda()
    m = tma()
    rng = np.random.default_rng(300 + seed)
    seqs = synth.random_sequences(rng, 40, 60, vocab=3, min_len=1)
    pk = _run(m, seqs, C, K, bf16, seed)
    assert pk["T"] > 100


def test_conv1d_tiny_tree_fp32():
    need_cuda()
    m = tma()
    _run(m, synth.tiny_tree().seqs, 64, 4, False, 0)


def test_conv1d_wide_fork_and_chain():
    """A root with 40 one- and two-token children (a wide fork inside one tile), then a
    long chain through several tiles; no bias."""
    need_cuda()
    m = tma()
    seqs = [[0, 1000 + i] + ([2000 + i] if i % 2 else []) for i in range(40)] + [[0] + list(range(1, 400))]
    _run(m, seqs, 32, 4, True, 9, bias=False)


def test_conv1d_galton_watson_full_size():
    """The 16384-row Galton-Watson tree at 8192 channels and K = 4 (bf16), the size the
    benchmark times; the oracle checks two 64-channel slices (channels are independent)."""
    need_cuda()
    m = tma()
    t = synth.galton_watson()
    cs = np.r_[0:64, 8128:8192]
    _run(m, t.seqs, 8192, 4, True, 11, channels=cs)


def test_conv1d_edge_cases():
    need_cuda()
    m = tma()
    # one row: y = w[:, K-1] x + b; dx = w[:, K-1] dy
    _run(m, [[5]], 8, 3, False, 2)
    # empty tree: nothing to do, dw and dbias are zero
    x = torch.empty((0, 16), dtype=torch.float32, device="cuda")
    w = torch.ones((16, 4), dtype=torch.float32, device="cuda")
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    y = m.tree_conv1d_fwd(x, w, e)
    dx, dw, db = m.tree_conv1d_bwd(x, w, x, e, e)
    assert y.shape == (0, 16) and float(dw.abs().sum()) == 0.0 and float(db.abs().sum()) == 0.0
    m.tree_check_device_status()


def test_conv1d_bad_parent_sets_device_flag():
    """A parent_row entry that is not an earlier row is reported through the device error
    word and read as 'no parent'; every index the kernel uses stays inside the tree."""
    need_cuda()
    m = tma()
    T = 100
    parent = np.arange(-1, T - 1, dtype=np.int32)
    parent[40] = 70
    x = torch.ones((T, 8), dtype=torch.float32, device="cuda")
    w = torch.ones((8, 2), dtype=torch.float32, device="cuda")
    y = m.tree_conv1d_fwd(x, w, dev(parent))
    with pytest.raises(m.TreeError) as ei:
        m.tree_check_device_status()
    assert ei.value.status == 7
    assert float(host(y)[40, 0]) == 1.0 and float(host(y)[41, 0]) == 2.0
    m.tree_check_device_status()   # cleared
