"""Pins for the CPU oracle: each checks it against something other than itself.

* library routines: torch fp64 SiLU / Linear / depthwise conv1d / rms_norm;
* brute force: per-token scalar Python loops on tiny shapes;
* closed forms: eta = 0, one chunk, and the associative (prefix) form of the
  pages' context-parallel algorithm, which never materialises W_c;
* invariants: affine in eta, reset, no cross-chunk leakage, row separability.

A planted-mistake test at the end swaps single steps of the oracle for
plausible wrong versions and checks that some pin fails for each.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.ttt_oracle as orc
from ttt_inputs import make_layer, round_bf16

TORCH64 = torch.float64


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def _tiny(d=4, f=8, T=13, C=4, k=2, eta=0.3, seed=3, doc_starts=(0,)):
    return make_layer(d, f, T, C, k, eta, dtype="f32", seed=seed, init="tiny",
                      doc_starts=doc_starts)


def _run(cfg, **kw):
    args = dict(eta=cfg["eta"], chunk=cfg["chunk"], doc_starts=cfg["doc_starts"])
    args.update(kw)
    return orc.ttt_layer(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"],
                         cfg["conv_w"], cfg["w_target"], **args)


# ---------------------------------------------------------------- library routines

def test_silu_matches_torch():
    a = np.linspace(-30, 30, 2001)
    np.testing.assert_allclose(orc.silu(a), F.silu(_t(a)).numpy(), rtol=1e-15, atol=1e-300)


def _torch_static_mlp(x, wg, wu, wd):
    x = _t(x)
    return F.linear(F.silu(F.linear(x, _t(wg))) * F.linear(x, _t(wu)), _t(wd)).numpy()


def test_swiglu_matches_torch_mlp():
    cfg = _tiny(d=16, f=40, T=7)
    z = orc.swiglu_intermediate(cfg["x"], cfg["w_gate"], cfg["w_up"])
    ref = _torch_static_mlp(cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"])
    assert _rel(z @ np.float64(cfg["w_down0"]).T, ref) < 1e-14


def _torch_target_source(x0_chunk, conv_w):
    """Depthwise conv1d (library) on the chunk shifted left by one token and
    zero-padded at its end: out[t] = sum_j w[j] * x0[t+1+j] inside the chunk."""
    x0 = _t(x0_chunk)
    n, d = x0.shape
    k = conv_w.shape[0]
    shifted = torch.zeros((n + k, d), dtype=TORCH64)
    shifted[: n - 1] = x0[1:]
    inp = shifted.T.unsqueeze(0)                       # 1 x d x (n+k)
    w = _t(conv_w).T.unsqueeze(1)                      # d x 1 x k
    out = F.conv1d(inp, w, groups=d)                   # 1 x d x (n+1)
    return out[0, :, :n].T.numpy()


@pytest.mark.parametrize("k", [1, 2, 4, 5, 8])
@pytest.mark.parametrize("n", [1, 2, 3, 9])
def test_conv_matches_torch_conv1d(k, n):
    rng = np.random.default_rng(k * 10 + n)
    x0 = rng.standard_normal((n, 6))
    cw = rng.standard_normal((k, 6))
    np.testing.assert_allclose(orc.chunk_target_source(x0, cw), _torch_target_source(x0, cw),
                               rtol=1e-13, atol=1e-13)


def _torch_target_source_mode(x0_chunk, conv_w, mode):
    """Library conv1d for the other windows: mode 1 (X0[t+j]) is conv1d on the
    chunk zero-padded at its end; mode 2 (X0[t+1-j]) is conv1d with the taps
    reversed over the chunk zero-padded on both sides (k zeros before, 2
    after), read at output t+2."""
    x0 = _t(x0_chunk)
    n, d = x0.shape
    k = conv_w.shape[0]
    w = _t(conv_w)
    if mode == 1:
        seq = torch.cat([x0, torch.zeros((k, d), dtype=TORCH64)])
        out = F.conv1d(seq.T.unsqueeze(0), w.T.unsqueeze(1), groups=d)
        return out[0, :, :n].T.numpy()
    seq = torch.cat([torch.zeros((k, d), dtype=TORCH64), x0, torch.zeros((2, d), dtype=TORCH64)])
    out = F.conv1d(seq.T.unsqueeze(0), w.flip(0).T.unsqueeze(1), groups=d)
    return out[0, :, 2:n + 2].T.numpy()


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("k", [1, 2, 5, 8])
@pytest.mark.parametrize("n", [1, 3, 9])
def test_target_modes_match_torch_conv1d(mode, k, n):
    rng = np.random.default_rng(100 * mode + 10 * k + n)
    x0 = rng.standard_normal((n, 5))
    cw = rng.standard_normal((k, 5))
    np.testing.assert_allclose(orc.chunk_target_source(x0, cw, mode),
                               _torch_target_source_mode(x0, cw, mode), rtol=1e-13, atol=1e-13)


def test_current_window_k1_is_reconstruction_target():
    rng = np.random.default_rng(4)
    x0 = rng.standard_normal((6, 3))
    cw = rng.standard_normal((1, 3))
    wt = rng.standard_normal((3, 3))
    v = orc.chunk_target(x0, cw, wt, orc.TARGET_CURRENT)
    np.testing.assert_allclose(v, (cw[0] * x0) @ wt, rtol=1e-14)


def test_causal_and_next_windows_agree_for_one_tap():
    rng = np.random.default_rng(5)
    x0 = rng.standard_normal((7, 4))
    cw = rng.standard_normal((1, 4))
    np.testing.assert_array_equal(orc.chunk_target_source(x0, cw, orc.TARGET_CAUSAL),
                                  orc.chunk_target_source(x0, cw, orc.TARGET_NEXT))


def test_k1_is_next_token_target():
    rng = np.random.default_rng(0)
    x0 = rng.standard_normal((5, 3))
    cw = rng.standard_normal((1, 3))
    wt = rng.standard_normal((3, 3))
    v = orc.chunk_target(x0, cw, wt)
    for t in range(4):
        np.testing.assert_allclose(v[t], (cw[0] * x0[t + 1]) @ wt, rtol=1e-14)
    assert np.all(v[4] == 0.0)  # the chunk's last token has no future token inside the chunk


def test_rms_norm_matches_torch():
    h = np.random.default_rng(1).standard_normal((9, 33)) * 3
    ref = F.rms_norm(_t(h), (33,), eps=1e-6).numpy()
    np.testing.assert_allclose(orc.rms_norm(h, 1e-6), ref, rtol=1e-14)


# ---------------------------------------------------------------- chunking

def test_chunk_spans_hand_written():
    assert orc.chunk_spans(10, 4) == [(0, 4, True), (4, 8, False), (8, 10, False)]
    assert orc.chunk_spans(10, 4, doc_starts=()) == [(0, 4, False), (4, 8, False), (8, 10, False)]
    # a document starting mid-chunk restarts the chunking there
    assert orc.chunk_spans(11, 4, doc_starts=(0, 6)) == [
        (0, 4, True), (4, 6, False), (6, 10, True), (10, 11, False)]
    assert orc.chunk_spans(3, 8) == [(0, 3, True)]
    assert orc.chunk_spans(0, 8, doc_starts=()) == []
    with pytest.raises(ValueError):
        orc.chunk_spans(5, 2, doc_starts=(5,))


# ---------------------------------------------------------------- brute force

def _silu_scalar(a):
    return a / (1.0 + math.exp(-a))


def brute_force_layer(x, x0, wg, wu, w0, cw, wt, eta, C, doc_starts=(0,), mode=0, tau=None):
    """Scalar, per-token restatement of the whole method (tiny shapes only).
    mode: target window (0: X0[t+1+j], 1: X0[t+j], 2: X0[t+1-j]); tau: clip
    each chunk's delta to Frobenius norm tau."""
    x = np.asarray(x, np.float64).tolist()
    x0 = np.asarray(x0, np.float64).tolist()
    wg = np.asarray(wg, np.float64).tolist()
    wu = np.asarray(wu, np.float64).tolist()
    w0 = np.asarray(w0, np.float64).tolist()
    cw = np.asarray(cw, np.float64).tolist()
    wt = np.asarray(wt, np.float64).tolist()
    n, d, f, k = len(x), len(x[0]), len(wg), len(cw)
    starts = sorted(doc_starts)
    W = [row[:] for row in w0]
    out = [[0.0] * d for _ in range(n)]
    t = 0
    while t < n:
        if t in starts:
            W = [row[:] for row in w0]
        nxt = [s for s in starts if s > t]
        e = min(t + C, n, nxt[0] if nxt else n)
        zs = []
        for i in range(t, e):
            z = []
            for p in range(f):
                g = sum(x[i][a] * wg[p][a] for a in range(d))
                u = sum(x[i][a] * wu[p][a] for a in range(d))
                z.append(_silu_scalar(g) * u)
            zs.append(z)
            for r in range(d):
                out[i][r] = sum(z[p] * W[r][p] for p in range(f))
        dW = [[0.0] * f for _ in range(d)]
        for i in range(t, e):
            src = [0.0] * d
            for j in range(k):
                s_tok = i + (1 + j, j, 1 - j)[mode]
                if t <= s_tok < e:
                    for a in range(d):
                        src[a] += cw[j][a] * x0[s_tok][a]
            for r in range(d):
                v = sum(src[a] * wt[a][r] for a in range(d))
                for p in range(f):
                    dW[r][p] += v * zs[i - t][p]
        scale = eta
        if tau:
            nrm = math.sqrt(sum((eta * dW[r][p]) ** 2 for r in range(d) for p in range(f)))
            if nrm > tau:
                scale = eta * tau / nrm
        for r in range(d):
            for p in range(f):
                W[r][p] += scale * dW[r][p]
        t = e
    return np.array(out), np.array(W)


BRUTE_CASES = [
    dict(T=13, C=4, k=1, doc_starts=(0,)),
    dict(T=13, C=4, k=2, doc_starts=(0,)),
    dict(T=13, C=4, k=5, doc_starts=(0,)),
    dict(T=13, C=3, k=2, doc_starts=(0, 5, 11)),
    dict(T=9, C=1, k=2, doc_starts=(0,)),
    dict(T=6, C=16, k=3, doc_starts=(0,)),
]


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_brute_force_tiny(case):
    cfg = _tiny(T=case["T"], C=case["C"], k=case["k"], doc_starts=case["doc_starts"])
    o, w = _run(cfg)
    ob, wb = brute_force_layer(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"],
                               cfg["conv_w"], cfg["w_target"], cfg["eta"], cfg["chunk"],
                               cfg["doc_starts"])
    assert _rel(o, ob) < 1e-12
    assert _rel(w, wb) < 1e-12


def _torch_intermediates(cfg):
    """Z from torch's Linear and SiLU, and V chunk by chunk from torch's
    depthwise conv1d and a matmul, over the chunks the call makes."""
    x = _t(cfg["x"])
    z = (F.silu(F.linear(x, _t(cfg["w_gate"]))) * F.linear(x, _t(cfg["w_up"]))).numpy()
    v = np.zeros((x.shape[0], cfg["d"]))
    cuts = sorted(set(cfg["doc_starts"]) | {0, cfg["T"]})
    for a, b in zip(cuts[:-1], cuts[1:]):
        for s in range(a, b, cfg["chunk"]):
            e = min(s + cfg["chunk"], b)
            v[s:e] = _torch_target_source(cfg["x0"][s:e], cfg["conv_w"]) @ np.float64(cfg["w_target"])
    return z, v


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_core_recursion_matches_brute_force(case):
    """The apply+update recursion on library-computed Z and V equals the
    scalar restatement of the whole method."""
    cfg = _tiny(T=case["T"], C=case["C"], k=case["k"], doc_starts=case["doc_starts"])
    z, v = _torch_intermediates(cfg)
    o, w = orc.ttt_core(z, v, cfg["w_down0"], cfg["eta"], cfg["chunk"], cfg["doc_starts"])
    ob, wb = brute_force_layer(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"],
                               cfg["conv_w"], cfg["w_target"], cfg["eta"], cfg["chunk"],
                               cfg["doc_starts"])
    assert _rel(o, ob) < 1e-12
    assert _rel(w, wb) < 1e-12


@pytest.mark.parametrize("mode,tau", [(1, None), (2, None), (0, 0.05), (2, 0.02), (1, 1e9)])
def test_brute_force_target_modes_and_clipping(mode, tau):
    cfg = _tiny(T=13, C=4, k=3, doc_starts=(0, 9), eta=0.8)
    o, w = _run(cfg, target_mode=mode, clip_tau=tau)
    ob, wb = brute_force_layer(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"],
                               cfg["conv_w"], cfg["w_target"], cfg["eta"], cfg["chunk"],
                               cfg["doc_starts"], mode=mode, tau=tau)
    assert _rel(o, ob) < 1e-12
    assert _rel(w, wb) < 1e-12


def test_brute_force_continuation_from_state():
    """A call that does not start a document continues from the given state."""
    cfg = _tiny(T=12, C=4, k=2)
    o_all, w_all = _run(cfg, doc_starts=(0,))
    sub = {k: (v[8:] if k in ("x", "x0") else v) for k, v in cfg.items()}
    _, w8 = _run({**cfg, "x": cfg["x"][:8], "x0": cfg["x0"][:8]})
    o2, w2 = _run(sub, doc_starts=(), w_init=w8)
    assert _rel(o2, o_all[8:]) < 1e-13 and _rel(w2, w_all) < 1e-13


# ---------------------------------------------------------------- closed forms

def test_eta_zero_is_static_mlp():
    cfg = _tiny(d=8, f=24, T=40, C=8, k=3)
    o, w = _run(cfg, eta=0.0)
    ref = _torch_static_mlp(cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"])
    assert _rel(o, ref) < 1e-14
    assert np.array_equal(w, np.float64(cfg["w_down0"]))


@pytest.mark.parametrize("zeroed", ["conv_w", "w_target"])
def test_zero_target_is_static_mlp(zeroed):
    """A zero conv or a zero target projection makes every V zero ("In-Place
    Test-Time Training" summary page, section 3, LM-Aligned Objective: the
    target is Conv1D(X0) W_target): the layer is the static MLP for any eta and
    W stays W_0 exactly."""
    cfg = _tiny(d=8, f=24, T=40, C=8, k=3)
    cfg = {**cfg, zeroed: np.zeros_like(cfg[zeroed])}
    o, w = _run(cfg, eta=0.5)
    ref = _torch_static_mlp(cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"])
    assert _rel(o, ref) < 1e-14
    assert np.array_equal(w, np.float64(cfg["w_down0"]))


def test_single_chunk_apply_before_update():
    """T <= C: the output is the static MLP for any eta; W_final = W_0 + eta V^T Z."""
    cfg = _tiny(d=8, f=24, T=10, C=16, k=3, eta=5.0)
    o, w = _run(cfg)
    ref = _torch_static_mlp(cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"])
    assert _rel(o, ref) < 1e-14
    x = _t(cfg["x"])
    z = F.silu(F.linear(x, _t(cfg["w_gate"]))) * F.linear(x, _t(cfg["w_up"]))
    v = _t(_torch_target_source(cfg["x0"], cfg["conv_w"])) @ _t(cfg["w_target"])
    w_ref = _t(cfg["w_down0"]) + cfg["eta"] * v.T @ z
    assert _rel(w, w_ref.numpy()) < 1e-14


def _prefix_form(cfg):
    """Associative form of the pages' context-parallel algorithm: with deltas
    D_j = eta V_j^T Z_j, chunk c uses W_0 + sum_{j<c} D_j, so
    O_c = Z_c W_0^T + eta sum_{j<c} (Z_c Z_j^T) V_j  (W_c never formed), and
    W_final = W_0 + sum_j D_j.  Z and V come from torch library ops."""
    x = _t(cfg["x"])
    z = F.silu(F.linear(x, _t(cfg["w_gate"]))) * F.linear(x, _t(cfg["w_up"]))
    C, T = cfg["chunk"], x.shape[0]
    spans = [(s, min(s + C, T)) for s in range(0, T, C)]
    v = torch.cat([_t(_torch_target_source(cfg["x0"][s:e], cfg["conv_w"])) for s, e in spans])
    v = v @ _t(cfg["w_target"])
    w0 = _t(cfg["w_down0"])
    out = torch.zeros((T, w0.shape[0]), dtype=TORCH64)
    for c, (s, e) in enumerate(spans):
        acc = z[s:e] @ w0.T
        for (s2, e2) in spans[:c]:
            acc = acc + cfg["eta"] * (z[s:e] @ z[s2:e2].T) @ v[s2:e2]
        out[s:e] = acc
    w_final = w0 + cfg["eta"] * v.T @ z
    return out.numpy(), w_final.numpy()


@pytest.mark.parametrize("T,C", [(64, 8), (50, 7), (32, 32), (33, 32)])
def test_recurrence_equals_prefix_form(T, C):
    cfg = _tiny(d=8, f=20, T=T, C=C, k=4, eta=0.7, seed=T)
    o, w = _run(cfg)
    op, wp = _prefix_form(cfg)
    assert _rel(o, op) < 1e-12
    assert _rel(w, wp) < 1e-12
    # the update term is not negligible in these cases
    o0, _ = _run(cfg, eta=0.0)
    if T > C:
        assert _rel(o, o0) > 1e-3


def test_clipping_bounds_every_chunk_delta():
    """With clipping, each chunk's delta keeps its direction and has norm
    min(||unclipped||, tau); a huge tau changes nothing."""
    cfg = _tiny(d=8, f=20, T=40, C=8, k=3, eta=0.9)
    tau = 0.05
    W = np.float64(cfg["w_down0"])
    for s, e, _ in orc.chunk_spans(cfg["T"], cfg["chunk"], (0,)):
        sub = {**cfg, "x": cfg["x"][s:e], "x0": cfg["x0"][s:e]}
        _, w_free = _run(sub, doc_starts=(), w_init=W)
        _, w_clip = _run(sub, doc_starts=(), w_init=W, clip_tau=tau)
        d_free, d_clip = w_free - W, w_clip - W
        n_free = np.linalg.norm(d_free)
        assert np.linalg.norm(d_clip) <= min(n_free, tau) * (1 + 1e-12)
        if n_free > tau:
            assert abs(np.linalg.norm(d_clip) - tau) <= 1e-12 * tau
            np.testing.assert_allclose(d_clip * n_free / tau, d_free, rtol=1e-10, atol=1e-14)
        W = w_clip
    o1, w1 = _run(cfg)
    o2, w2 = _run(cfg, clip_tau=1e12)
    assert np.array_equal(o1, o2) and np.array_equal(w1, w2)


def test_chunk_delta_norms_are_the_recursions_deltas():
    cfg = _tiny(d=8, f=20, T=30, C=7, k=3, doc_starts=(0, 16))
    norms = orc.chunk_delta_norms(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"], cfg["conv_w"],
                                  cfg["w_target"], cfg["eta"], cfg["chunk"], cfg["doc_starts"])
    spans = orc.chunk_spans(cfg["T"], cfg["chunk"], cfg["doc_starts"])
    assert len(norms) == len(spans)
    W = np.float64(cfg["w_down0"])
    for (s, e, reset), nrm in zip(spans, norms):
        if reset:
            W = np.float64(cfg["w_down0"])
        sub = {**cfg, "x": cfg["x"][s:e], "x0": cfg["x0"][s:e]}
        _, w_next = _run(sub, doc_starts=(), w_init=W)
        assert abs(np.linalg.norm(w_next - W) - nrm) <= 1e-12 * max(nrm, 1e-300)
        W = w_next


def test_gram_identity_for_the_update_norm():
    """||V^T Z||_F^2 = <V V^T, Z Z^T>_F (the form the kernels use to get a
    chunk's delta norm without forming the delta), checked with torch."""
    rng = np.random.default_rng(9)
    v = _t(rng.standard_normal((16, 7)))
    z = _t(rng.standard_normal((16, 11)))
    lhs = torch.linalg.matrix_norm(v.T @ z) ** 2
    rhs = torch.sum((v @ v.T) * (z @ z.T))
    assert abs(float(lhs - rhs)) <= 1e-12 * float(lhs)


def test_affine_in_eta():
    cfg = _tiny(d=8, f=20, T=48, C=8, k=3)
    o0, w0 = _run(cfg, eta=0.0)
    o1, w1 = _run(cfg, eta=0.4)
    o2, w2 = _run(cfg, eta=0.8)
    assert np.max(np.abs(o2 - 2 * o1 + o0)) <= 1e-12 * np.max(np.abs(o1))
    assert np.max(np.abs(w2 - 2 * w1 + w0)) <= 1e-12 * np.max(np.abs(w1))
    assert _rel(o1, o0) > 1e-3


# ---------------------------------------------------------------- invariants

def test_reset_matches_documents_run_alone():
    cfg = _tiny(d=8, f=20, T=40, C=6, k=3, doc_starts=(0, 17, 29))
    o, w = _run(cfg)
    bounds = [(0, 17), (17, 29), (29, 40)]
    for s, e in bounds:
        sub = {**cfg, "x": cfg["x"][s:e], "x0": cfg["x0"][s:e]}
        os_, ws = _run(sub, doc_starts=(0,))
        assert np.array_equal(o[s:e], os_)
    assert np.array_equal(w, ws)  # final W = last document's own final W


def test_no_cross_chunk_target_leakage():
    cfg = _tiny(d=8, f=20, T=40, C=8, k=5)
    o, _ = _run(cfg)
    x0 = cfg["x0"].copy()
    x0[16:24] += 1.0  # perturb chunk 2's embeddings only
    o2, _ = _run({**cfg, "x0": x0})
    assert np.array_equal(o[:24], o2[:24])   # chunks 0..2 use W_0 + D_0 + D_1 only
    assert not np.array_equal(o[24:32], o2[24:32])  # chunk 3 sees D_2


def test_row_sampled_equals_full():
    cfg = _tiny(d=12, f=20, T=30, C=7, k=3, doc_starts=(0, 11))
    o, w = _run(cfg)
    rows = [0, 5, 11, 3]
    orow, wrow = orc.ttt_layer_rows(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"],
                                    cfg["w_down0"], cfg["conv_w"], cfg["w_target"], cfg["eta"],
                                    cfg["chunk"], rows, cfg["doc_starts"])
    assert _rel(orow, o[:, rows]) < 1e-13
    assert _rel(wrow, w[rows]) < 1e-13
    # a precomputed Z (from the torch library MLP) gives the same rows
    x = _t(cfg["x"])
    z = (F.silu(F.linear(x, _t(cfg["w_gate"]))) * F.linear(x, _t(cfg["w_up"]))).numpy()
    orow2, wrow2 = orc.ttt_layer_rows(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"],
                                      cfg["w_down0"], cfg["conv_w"], cfg["w_target"], cfg["eta"],
                                      cfg["chunk"], rows, cfg["doc_starts"], z=z)
    assert _rel(orow2, o[:, rows]) < 1e-13
    assert _rel(wrow2, w[rows]) < 1e-13
    # other target windows and clipping: rows still equal the full recursion
    for mode, tau in ((2, 0.01), (1, None)):
        o3, w3 = _run(cfg, target_mode=mode, clip_tau=tau)
        orow3, wrow3 = orc.ttt_layer_rows(cfg["x"], cfg["x0"], cfg["w_gate"], cfg["w_up"],
                                          cfg["w_down0"], cfg["conv_w"], cfg["w_target"],
                                          cfg["eta"], cfg["chunk"], rows, cfg["doc_starts"],
                                          target_mode=mode, clip_tau=tau)
        assert _rel(orow3, o3[:, rows]) < 1e-13
        assert _rel(wrow3, w3[rows]) < 1e-13


def test_stack_matches_brute_force_composition():
    from ttt_inputs import make_stack
    h0, layers, meta = make_stack(3, 4, 8, 10, 4, 2, 0.5, seed=2, dtype="f32")
    h, finals = orc.ttt_stack(h0, layers, meta["eta"], meta["chunk"])
    hb = np.float64(h0)
    for li, w in enumerate(layers):
        xn = F.rms_norm(_t(hb), (hb.shape[1],), eps=1e-6).numpy()
        ob, wb = brute_force_layer(xn, h0, w["w_gate"], w["w_up"], w["w_down0"], w["conv_w"],
                                   w["w_target"], meta["eta"], meta["chunk"])
        hb = hb + ob
        assert _rel(finals[li], wb) < 1e-12
    assert _rel(h, hb) < 1e-12


@pytest.mark.parametrize("every", [1, 2, 3])
def test_stack_placement_matches_brute_force_composition(every):
    """TTT in every `every`-th block (1-based), the others the plain SwiGLU
    MLP: brute force for the TTT blocks and torch's Linear/SiLU MLP for the
    static ones, composed with torch's rms_norm."""
    from ttt_inputs import make_stack
    h0, layers, meta = make_stack(4, 4, 8, 10, 4, 2, 0.5, seed=5, dtype="f32")
    h, finals = orc.ttt_stack(h0, layers, meta["eta"], meta["chunk"], ttt_every=every)
    hb = np.float64(h0)
    for li, w in enumerate(layers):
        xn = F.rms_norm(_t(hb), (hb.shape[1],), eps=1e-6).numpy()
        if (li + 1) % every == 0:
            ob, wb = brute_force_layer(xn, h0, w["w_gate"], w["w_up"], w["w_down0"], w["conv_w"],
                                       w["w_target"], meta["eta"], meta["chunk"])
        else:
            ob, wb = _torch_static_mlp(xn, w["w_gate"], w["w_up"], w["w_down0"]), w["w_down0"]
        hb = hb + ob
        assert _rel(finals[li], wb) < 1e-12
    assert _rel(h, hb) < 1e-12
    if every == 1:
        h1, _ = orc.ttt_stack(h0, layers, meta["eta"], meta["chunk"])
        assert np.array_equal(h, h1)
    # the per-block states: h_0 = h0, h_L = the result, and each step is the
    # block output of the brute-force composition above
    _, _, states = orc.ttt_stack(h0, layers, meta["eta"], meta["chunk"], ttt_every=every,
                                 return_states=True)
    assert len(states) == len(layers) + 1
    assert np.array_equal(states[0], np.float64(h0)) and np.array_equal(states[-1], h)
    hb = np.float64(h0)
    for li, w in enumerate(layers):
        xn = F.rms_norm(_t(hb), (hb.shape[1],), eps=1e-6).numpy()
        if (li + 1) % every == 0:
            ob, _ = brute_force_layer(xn, h0, w["w_gate"], w["w_up"], w["w_down0"], w["conv_w"],
                                      w["w_target"], meta["eta"], meta["chunk"])
        else:
            ob = _torch_static_mlp(xn, w["w_gate"], w["w_up"], w["w_down0"])
        assert _rel(states[li + 1], hb + ob) < 1e-12
        hb = hb + ob


def test_static_mlp_matches_torch_and_eta_zero_layer():
    cfg = _tiny(d=8, f=24, T=11, C=4, k=3)
    ref = _torch_static_mlp(cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"])
    o = orc.static_mlp(cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"])
    assert _rel(o, ref) < 1e-14
    o0, _ = _run(cfg, eta=0.0)
    assert _rel(o, o0) < 1e-14


def test_bf16_inputs_are_exact_in_oracle():
    """The oracle sees exactly the stored (bf16-rounded) input values."""
    cfg = make_layer(16, 32, 8, 4, 2, 1e-3, dtype="bf16", init="qwen")
    assert np.array_equal(round_bf16(cfg["x"]), cfg["x"])
    assert np.array_equal(round_bf16(cfg["w_gate"]), cfg["w_gate"])


# ---------------------------------------------------------------- planted mistakes

def _pins_pass(module_overrides):
    """Run a subset of the pins above with oracle functions replaced."""
    saved = {k: getattr(orc, k) for k in module_overrides}
    try:
        for k, v in module_overrides.items():
            setattr(orc, k, v)
        checks = [
            lambda: test_brute_force_tiny(BRUTE_CASES[1]),
            lambda: test_brute_force_tiny(BRUTE_CASES[3]),
            lambda: test_single_chunk_apply_before_update(),
            lambda: test_recurrence_equals_prefix_form(50, 7),
            lambda: test_no_cross_chunk_target_leakage(),
            lambda: test_reset_matches_documents_run_alone(),
            lambda: test_brute_force_target_modes_and_clipping(0, 0.05),
            lambda: test_brute_force_target_modes_and_clipping(2, None),
            lambda: test_target_modes_match_torch_conv1d(2, 5, 9),
            lambda: test_core_recursion_matches_brute_force(BRUTE_CASES[3]),
            lambda: test_stack_placement_matches_brute_force_composition(3),
        ]
        for c in checks:
            try:
                c()
            except AssertionError:
                return False
        return True
    finally:
        for k, v in saved.items():
            setattr(orc, k, v)


def _update_before_apply(x, x0, w_gate, w_up, w_down0, conv_w, w_target, eta, chunk,
                         doc_starts=(0,), w_init=None):
    x, x0, w0 = map(np.float64, (x, x0, w_down0))
    W = w0.copy()
    out = np.zeros((x.shape[0], w0.shape[0]))
    for s, e, reset in orc.chunk_spans(x.shape[0], chunk, doc_starts):
        if reset:
            W = w0.copy()
        z = orc.swiglu_intermediate(x[s:e], w_gate, w_up)
        W = W + eta * (orc.chunk_target(x0[s:e], conv_w, w_target).T @ z)
        out[s:e] = z @ W.T
    return out, W


def _core_update_before_apply(z, v, w_down0, eta, chunk, doc_starts=(0,), w_init=None):
    z, v, w0 = map(np.float64, (z, v, w_down0))
    W = w0.copy()
    out = np.zeros((z.shape[0], w0.shape[0]))
    for s, e, reset in orc.chunk_spans(z.shape[0], chunk, doc_starts):
        if reset:
            W = w0.copy()
        W = W + eta * (v[s:e].T @ z[s:e])
        out[s:e] = z[s:e] @ W.T
    return out, W


def _core_misaligned_update(z, v, w_down0, eta, chunk, doc_starts=(0,), w_init=None):
    # each token's Z paired with another token's target (rows reversed in the chunk)
    z, v, w0 = map(np.float64, (z, v, w_down0))
    W = w0.copy()
    out = np.zeros((z.shape[0], w0.shape[0]))
    for s, e, reset in orc.chunk_spans(z.shape[0], chunk, doc_starts):
        if reset:
            W = w0.copy()
        out[s:e] = z[s:e] @ W.T
        W = W + eta * (v[s:e][::-1].T @ z[s:e])
    return out, W


def _no_reset_spans(n, chunk, doc_starts=(0,)):
    return [(s, e, s == 0) for s, e, _ in _ORIG_SPANS(n, chunk, doc_starts)]


def _current_token_conv(x0_chunk, conv_w, mode=0):
    x0 = np.float64(x0_chunk)
    u = np.zeros_like(x0)
    for j in range(conv_w.shape[0]):
        m = x0.shape[0] - j
        if m > 0:
            u[:m] += np.float64(conv_w[j]) * x0[j:j + m]
    return u


def _leaky_conv(x0_chunk, conv_w, mode=0):
    # forgets the chunk-end padding: wraps around inside the chunk
    x0 = np.float64(x0_chunk)
    u = np.zeros_like(x0)
    for j in range(conv_w.shape[0]):
        u += np.float64(conv_w[j]) * np.roll(x0, -(1 + j), axis=0)
    return u


_ORIG_SPANS = orc.chunk_spans
_ORIG_TARGET = orc.chunk_target
_ORIG_SOURCE = orc.chunk_target_source


def _causal_off_by_one(x0_chunk, conv_w, mode=0):
    # the causal window ending at the current token instead of the next one
    return _ORIG_SOURCE(x0_chunk, conv_w, 1 if mode == 2 else mode) if mode != 2 else \
        np.vstack([np.zeros((1, np.shape(x0_chunk)[1])),
                   _ORIG_SOURCE(x0_chunk, conv_w, 2)[:-1]])


def _clip_by_max(delta, tau):
    m = float(np.max(np.abs(delta)))
    return delta * (tau / m) if tau and m > tau else delta


def _stack_placement_from_zero(h0, layers, eta, chunk, doc_starts=(0,), eps=1e-6, n_layers=None,
                               x0=None, target_mode=0, clip_tau=None, ttt_every=1):
    # TTT in blocks 0, s, 2s, ... instead of the s-th, 2s-th, ... (1-based)
    h = np.float64(h0).copy()
    finals = []
    for li, w in enumerate(layers[: n_layers or len(layers)]):
        xn = orc.rms_norm(h, eps)
        if li % ttt_every == 0:
            o, wf = orc.ttt_layer(xn, np.float64(h0), w["w_gate"], w["w_up"], w["w_down0"],
                                  w["conv_w"], w["w_target"], eta, chunk, doc_starts)
        else:
            o, wf = orc.static_mlp(xn, w["w_gate"], w["w_up"], w["w_down0"]), np.float64(w["w_down0"])
        h = h + o
        finals.append(wf)
    return h, finals


def test_planted_mistakes_are_caught():
    assert _pins_pass({})
    mistakes = {
        "update before apply": {"ttt_layer": _update_before_apply},
        "no document reset": {"chunk_spans": _no_reset_spans},
        "target from the current token": {"chunk_target_source": _current_token_conv},
        "target wraps inside the chunk": {"chunk_target_source": _leaky_conv},
        "W_target transposed": {"chunk_target": lambda x0, cw, wt, mode=0:
                                orc.chunk_target_source(x0, cw) @ np.float64(wt).T},
        "update sign flipped": {"chunk_target": lambda x0, cw, wt, mode=0: -_ORIG_TARGET(x0, cw, wt)},
        "SiLU sign flipped": {"silu": lambda a: np.float64(a) / (1 + np.exp(np.float64(a)))},
        "clipping ignored": {"clip_delta": lambda delta, tau: delta},
        "clipping by max-abs, not Frobenius": {"clip_delta": _clip_by_max},
        "causal window shifted by one token": {"chunk_target_source": _causal_off_by_one},
        "core: update before apply": {"ttt_core": _core_update_before_apply},
        "placement counted from block 0": {"ttt_stack": _stack_placement_from_zero},
        "core: a chunk's target rows paired with the wrong tokens": {"ttt_core": _core_misaligned_update},
    }
    for name, ov in mistakes.items():
        assert not _pins_pass(ov), f"planted mistake not caught: {name}"
