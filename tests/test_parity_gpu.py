"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle on
the same seeded inputs.

Tolerances (relative Frobenius error ||gpu - oracle|| / ||oracle||):
  * fp32 activations (FFMA path, no TF32):        1e-5 on O and on final W
  * bf16 activations / fp32 accumulation and W:    1e-2 on O and on final W
The bf16 path also reports the error of the TTT part alone, O - Z W_0^T, which
the static part would otherwise dominate; it must stay within 5e-2 (the bf16
roundings of Z, V, the Gram block and the W operand copy are each ~2^-9
relative; measured values are far below this bound).
"""
import os

import numpy as np
import pytest
import torch

import oracle.ttt_oracle as orc
from ttt_inputs import make_layer

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5
TOL_BF16 = 1e-2
TOL_TTT_PART = 5e-2


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device="cuda", dtype=dtype)


def _host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _make_gpu_layer(cfg, n_docs=1, max_tokens=None, dtype=None, **opts):
    from chunk_wise_weight_ttt_b300 import TTTMLP
    dt = dtype or (torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32)
    ws = [_dev(cfg[k], dt) for k in ("w_gate", "w_up", "w_down0", "conv_w", "w_target")]
    layer = TTTMLP(*ws, chunk=cfg["chunk"], eta=cfg["eta"], n_docs=n_docs,
                   max_tokens=max_tokens or cfg["T"], **opts)
    return layer, dt


def _oracle(cfg, eta=None, doc_starts=None, x=None, w_init=None, target_mode=0, clip_tau=None):
    x = cfg["x"] if x is None else x
    return orc.ttt_layer(x, x, cfg["w_gate"], cfg["w_up"], cfg["w_down0"], cfg["conv_w"],
                         cfg["w_target"], cfg["eta"] if eta is None else eta, cfg["chunk"],
                         cfg["doc_starts"] if doc_starts is None else doc_starts, w_init=w_init,
                         target_mode=target_mode, clip_tau=clip_tau)


def _check_layer(cfg, tol, ttt_tol=None, force_simt=False, expect_path=None, target_mode=0,
                 clip_tau=None):
    if force_simt:
        os.environ["TTT_FORCE_SIMT"] = "1"
    try:
        layer, dt = _make_gpu_layer(cfg, target_mode=target_mode, clip_tau=clip_tau or 0.0)
    finally:
        os.environ.pop("TTT_FORCE_SIMT", None)
    if expect_path:
        assert layer.path == expect_path
    x = _dev(cfg["x"], dt)
    o = layer.forward(x, doc_starts=cfg["doc_starts"])
    w = layer.get_fast_weight()
    layer.check()
    torch.cuda.synchronize()
    o_ref, w_ref = _oracle(cfg, target_mode=target_mode, clip_tau=clip_tau)
    eo, ew = _rel(_host(o), o_ref), _rel(_host(w), w_ref)
    msg = f"O err {eo:.3e}  W err {ew:.3e}"
    if ttt_tol is not None:
        o_static, _ = _oracle(cfg, eta=0.0)
        part_gpu, part_ref = _host(o) - o_static, o_ref - o_static
        frac = np.linalg.norm(part_ref) / np.linalg.norm(o_ref)
        if frac > 1e-6:  # a single chunk has no TTT part
            ep = _rel(part_gpu, part_ref)
            msg += f"  TTT-part err {ep:.3e} (TTT part is {frac:.1%} of O)"
            assert ep <= ttt_tol, msg
        else:
            msg += "  (no TTT part: one chunk)"
    print(msg)
    assert eo <= tol and ew <= tol, msg
    return layer


# ------------------------------------------------------------------ fp32 path

def test_tiny_fp32_config_full():
    """d=64, f=256, T=1024, C=64, k=4, eta=0.01, fp32 -- the tiny configuration."""
    cfg = make_layer(64, 256, 1024, 64, 4, 0.01, dtype="f32", seed=0, init="tiny")
    _check_layer(cfg, TOL_F32, expect_path="simt")


@pytest.mark.parametrize("T,C,k,starts", [(77, 16, 2, (0,)), (130, 7, 5, (0, 33, 100)),
                                          (64, 64, 1, (0,)), (5, 8, 3, (0,))])
def test_fp32_ragged(T, C, k, starts):
    cfg = make_layer(16, 40, T, C, k, 0.05, dtype="f32", seed=T, init="tiny", doc_starts=starts)
    _check_layer(cfg, TOL_F32, expect_path="simt")


# ------------------------------------------------------------------ bf16 tcgen05 path

def _bf16_cfg(d=256, f=512, T=1000, C=64, k=5, eta=0.5, seed=1, starts=(0,)):
    return make_layer(d, f, T, C, k, eta, dtype="bf16", seed=seed, init="qwen", doc_starts=starts)


def test_bf16_intermediates_z_and_v():
    """Producer outputs on their own: Z (SwiGLU) and V = eta Conv1D(X0) W_target."""
    cfg = _bf16_cfg(T=700, C=100)
    layer, dt = _make_gpu_layer(cfg)
    assert layer.path == "tcgen05"
    x = _dev(cfg["x"], dt)
    layer.forward(x, doc_starts=(0,))
    layer.check()
    z, v = layer.intermediates(cfg["T"])
    z_ref = orc.swiglu_intermediate(cfg["x"], cfg["w_gate"], cfg["w_up"])
    v_ref = np.concatenate([cfg["eta"] * orc.chunk_target(cfg["x"][s:e], cfg["conv_w"],
                                                          cfg["w_target"])
                            for s, e, _ in orc.chunk_spans(cfg["T"], cfg["chunk"], (0,))])
    ez, ev = _rel(_host(z), z_ref), _rel(_host(v), v_ref)
    print(f"Z err {ez:.3e}  V err {ev:.3e}")
    assert ez < 8e-3 and ev < 8e-3


@pytest.mark.parametrize("T,C,starts", [
    (1000, 64, (0,)),            # 16 chunks; groups of 16 chunks, ragged tail
    (1024, 256, (0,)),           # groups of 4 chunks
    (1536, 512, (0,)),           # groups of 2 chunks
    (2048, 1024, (0,)),          # one chunk per group
    (900, 100, (0,)),            # chunk not a multiple of the 64-token K block
    (1100, 128, (0, 300, 777)),  # document starts off the chunk grid
    (300, 40, (0, 1, 2, 150)),   # one-token documents
    (64, 256, (0,)),             # a single short chunk: static MLP
])
def test_bf16_tcgen05_parity(T, C, starts):
    cfg = _bf16_cfg(T=T, C=C, starts=starts, seed=T + C)
    _check_layer(cfg, TOL_BF16, ttt_tol=TOL_TTT_PART, expect_path="tcgen05")


@pytest.mark.parametrize("d,f,T,C,k,starts", [
    (320, 576, 700, 100, 5, (0,)),       # 3 row blocks of d (a pair with one tile out of range), ragged f
    (384, 320, 1030, 256, 8, (0, 515)),  # ragged f tile, 8 taps, a document start mid-group
    (256, 256, 513, 1, 3, (0,)),         # one-token chunks: no chunk has a target, W stays W_0
    (512, 1024, 2300, 512, 2, (0, 2047)),
])
def test_bf16_tcgen05_ragged_pairs(d, f, T, C, k, starts):
    cfg = make_layer(d, f, T, C, k, 0.5, dtype="bf16", seed=d + f + T, init="qwen",
                     doc_starts=starts)
    layer = _check_layer(cfg, TOL_BF16, ttt_tol=TOL_TTT_PART, expect_path="tcgen05")
    if C == 1:
        assert torch.equal(layer.get_fast_weight().cpu(),
                           torch.from_numpy(np.float32(cfg["w_down0"])))


# ------------------------------------------------------------------ chained group launches

# Documents of mixed lengths at d=256, f=512, C=64 (groups of 2048 tokens):
# twelve groups against six S slots (two waves); runs that end at groups whose
# length is not a whole number of 64-token K blocks (188, 324, 52 and 204
# tokens); a document start at every group, so every run has resets inside it.
CHAIN_STARTS = (0, 256, 512, 700, 1024, 1536, 2048, 2100, 2304, 2560, 3072, 3584)


def _chain_cfg():
    return make_layer(256, 512, 4096, 64, 4, 0.5, dtype="bf16", seed=77, init="qwen",
                      doc_starts=CHAIN_STARTS)


def _chain_run(path=None):
    """One forward call of the chained-group case; saves (O, W) when `path` is given."""
    cfg = _chain_cfg()
    layer, dt = _make_gpu_layer(cfg)
    o = layer.forward(_dev(cfg["x"], dt), doc_starts=cfg["doc_starts"])
    w = layer.get_fast_weight()
    layer.check()
    res = (o.cpu(), w.cpu())
    if path:
        torch.save(res, path)
    return res


def test_chained_groups_waves_runs_and_resets():
    _check_layer(_chain_cfg(), TOL_BF16, ttt_tol=TOL_TTT_PART, expect_path="tcgen05")


@pytest.mark.parametrize("run", ["1", "3"])
def test_chained_launch_equals_shorter_runs(tmp_path, run):
    """A tile does the same arithmetic whether its group shares a launch with
    others or not, so the default launch (every group of a wave chained) must
    equal runs of at most `run` groups (TTT_GROUP_RUN, read once per process,
    hence a child process) bit for bit."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = tmp_path / "short_runs.pt"
    env = dict(os.environ, TTT_GROUP_RUN=run,
               PYTHONPATH=os.pathsep.join([root, os.path.join(root, "tests")]))
    subprocess.run([sys.executable, "-c", f"import test_parity_gpu as t; t._chain_run({str(out)!r})"],
                   env=env, cwd=root, check=True, timeout=600)
    o_short, w_short = torch.load(out)
    o_long, w_long = _chain_run()
    assert torch.equal(o_long, o_short)
    assert torch.equal(w_long, w_short)


# ------------------------------------------------------------------ target windows, clipping

@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("path", ["tcgen05", "simt"])
def test_target_windows(mode, path):
    """The current-token and causal windows (k=5), on both kernel families."""
    if path == "tcgen05":
        cfg = _bf16_cfg(T=900, C=100, seed=mode)
        _check_layer(cfg, TOL_BF16, ttt_tol=TOL_TTT_PART, expect_path="tcgen05", target_mode=mode)
    else:
        cfg = make_layer(16, 40, 130, 7, 5, 0.05, dtype="f32", seed=mode, init="tiny",
                         doc_starts=(0, 33, 100))
        _check_layer(cfg, TOL_F32, expect_path="simt", target_mode=mode)


def test_reconstruction_target_one_tap():
    """k=1 with the current-token window is the canonical reconstruction target."""
    cfg = _bf16_cfg(T=700, C=64, k=1, seed=11)
    _check_layer(cfg, TOL_BF16, ttt_tol=TOL_TTT_PART, expect_path="tcgen05", target_mode=1)


def _median_tau(cfg, mode=0):
    norms = orc.chunk_delta_norms(cfg["x"], cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["conv_w"],
                                  cfg["w_target"], cfg["eta"], cfg["chunk"], cfg["doc_starts"],
                                  target_mode=mode)
    return float(np.median(norms[norms > 0]))


@pytest.mark.parametrize("T,C,starts,mode", [(1000, 64, (0,), 0), (1100, 128, (0, 300, 777), 2),
                                             (2048, 1024, (0,), 0), (1536, 512, (0, 700), 1)])
def test_update_clipping_tcgen05(T, C, starts, mode):
    """Per-chunk clipping with tau at the median chunk-delta norm: about half
    the chunks are clipped, so the clipped update is a large part of O."""
    cfg = _bf16_cfg(T=T, C=C, starts=starts, seed=T + C + 3)
    tau = _median_tau(cfg, mode)
    _check_layer(cfg, TOL_BF16, ttt_tol=TOL_TTT_PART, expect_path="tcgen05", target_mode=mode,
                 clip_tau=tau)


def test_update_clipping_simt_fp32():
    cfg = make_layer(16, 40, 130, 7, 5, 0.5, dtype="f32", seed=21, init="tiny",
                     doc_starts=(0, 33, 100))
    tau = _median_tau(cfg)
    _check_layer(cfg, TOL_F32, expect_path="simt", clip_tau=tau)


def test_update_clipping_at_the_pages_threshold():
    """tau = 1e-5 (the pages' long-context evaluation): every delta is clipped
    to norm 1e-5, only a few fp32 ulps of W per element.  The group's delta is
    accumulated from zero and added to W in one rounding, so the accumulated
    update W - W_0 itself matches the oracle's (bound 5e-2: fp32 W rounds each
    group's addition)."""
    cfg = _bf16_cfg(T=1024, C=128, seed=5)
    layer, dt = _make_gpu_layer(cfg, clip_tau=1e-5)
    o = layer.forward(_dev(cfg["x"], dt), doc_starts=(0,))
    w = _host(layer.get_fast_weight())
    layer.check()
    o_ref, w_ref = _oracle(cfg, clip_tau=1e-5)
    assert _rel(_host(o), o_ref) <= TOL_BF16 and _rel(w, w_ref) <= TOL_BF16
    w0 = np.float64(cfg["w_down0"])
    err = _rel(w - w0, w_ref - w0)
    cos = float(np.sum((w - w0) * (w_ref - w0)) /
                (np.linalg.norm(w - w0) * np.linalg.norm(w_ref - w0)))
    print(f"tau=1e-5: |W - W0| {np.linalg.norm(w_ref - w0):.3e}, W err {_rel(w, w_ref):.3e}, "
          f"error of W - W0 {err:.3e}, cosine {cos:.4f}")
    assert err <= 5e-2 and cos >= 0.999


def test_empty_call_and_token_limit():
    from chunk_wise_weight_ttt_b300 import TTTError
    cfg = _bf16_cfg(T=256, C=64)
    layer, dt = _make_gpu_layer(cfg)
    x = _dev(cfg["x"], dt)
    empty = x[:0]
    o = layer.forward(empty, doc_starts=())
    assert o.shape == (0, cfg["d"])
    assert np.array_equal(_host(layer.get_fast_weight()), np.float64(cfg["w_down0"]))
    big = torch.zeros((cfg["T"] + 1, cfg["d"]), dtype=dt, device="cuda")
    with pytest.raises(TTTError, match="EINVAL"):
        layer.forward(big)                             # one token over max_tokens
    o = layer.forward(x)                               # exactly max_tokens
    o_ref, _ = _oracle(cfg)
    assert _rel(_host(o), o_ref) < TOL_BF16
    layer.check()


def test_bf16_simt_path_parity():
    cfg = _bf16_cfg(T=500, C=64)
    _check_layer(cfg, TOL_BF16, ttt_tol=TOL_TTT_PART, force_simt=True, expect_path="simt")


def test_eta_zero_keeps_w0_bitwise():
    cfg = _bf16_cfg(T=600, C=64, eta=0.0)
    layer, dt = _make_gpu_layer(cfg)
    layer.forward(_dev(cfg["x"], dt))
    w = layer.get_fast_weight()
    torch.cuda.synchronize()
    assert np.array_equal(_host(w), np.float64(cfg["w_down0"]))


def test_zero_conv_keeps_w0_bitwise_for_any_eta():
    """With a zero conv every target is zero, so every update adds exact zeros:
    W stays W_0 bit for bit on the tcgen05 path, and O is the static MLP."""
    cfg = _bf16_cfg(T=1100, C=64, eta=0.5)
    cfg = {**cfg, "conv_w": np.zeros_like(cfg["conv_w"])}
    layer, dt = _make_gpu_layer(cfg)
    assert layer.path == "tcgen05"
    o = layer.forward(_dev(cfg["x"], dt))
    w = layer.get_fast_weight()
    layer.check()
    assert np.array_equal(_host(w), np.float64(cfg["w_down0"]))
    o_ref, _ = _oracle(cfg, eta=0.0)
    assert _rel(_host(o), o_ref) < TOL_BF16


@pytest.mark.parametrize("path,C", [("tcgen05", 64), ("tcgen05", 1024), ("simt", 64)])
def test_static_forward_is_the_plain_mlp(path, C):
    """ttt_mlp_forward_static: SwiGLU(X) W_0^T against the oracle's static
    MLP, on both kernel families; and the same values as a forward call with
    eta = 0 (whose updates add exact zeros)."""
    cfg = _bf16_cfg(T=777, C=C, eta=0.0)
    if path == "simt":
        os.environ["TTT_FORCE_SIMT"] = "1"
    try:
        layer, dt = _make_gpu_layer(cfg)
    finally:
        os.environ.pop("TTT_FORCE_SIMT", None)
    assert layer.path == path
    x = _dev(cfg["x"], dt)
    o = layer.forward_static(x)
    o_eta0 = layer.forward(x)
    w = layer.get_fast_weight()
    layer.check()
    ref = orc.static_mlp(cfg["x"], cfg["w_gate"], cfg["w_up"], cfg["w_down0"])
    e = _rel(_host(o), ref)
    e0 = _rel(_host(o), _host(o_eta0))
    print(f"{path} C={C}: static O err {e:.3e}; vs the eta=0 layer {e0:.3e} "
          f"(bitwise {torch.equal(o, o_eta0)})")
    assert e <= TOL_BF16
    assert e0 <= 1e-6
    assert np.array_equal(_host(w), np.float64(cfg["w_down0"]))


def test_handles_sharing_scratch_equal_private_workspaces():
    """Two layers with their own state and one shared scratch, called one
    after another on one stream (and interleaved across two calls each), give
    the same bits as two layers with private workspaces."""
    from chunk_wise_weight_ttt_b300 import TTTMLP, workspace_bytes
    cfgs = [_bf16_cfg(T=900, C=64, seed=s, starts=(0, 300)) for s in (11, 12)]
    dt = torch.bfloat16
    scratch = torch.empty(workspace_bytes(256, 512, chunk=64, conv_k=5, max_tokens=900,
                                          part="scratch"), dtype=torch.uint8, device="cuda")
    shared, private = [], []
    for cfg in cfgs:
        ws = [_dev(cfg[k], dt) for k in ("w_gate", "w_up", "w_down0", "conv_w", "w_target")]
        shared.append(TTTMLP(*ws, chunk=64, eta=cfg["eta"], max_tokens=900, scratch=scratch))
        private.append(TTTMLP(*ws, chunk=64, eta=cfg["eta"], max_tokens=900))
    xs = [_dev(cfg["x"], dt) for cfg in cfgs]
    outs = {}
    for rnd in range(2):
        for i in range(2):
            starts = (0, 300) if rnd == 0 else ()
            outs[("s", rnd, i)] = shared[i].forward(xs[i], doc_starts=starts).clone()
            outs[("p", rnd, i)] = private[i].forward(xs[i], doc_starts=starts)
    for l in shared + private:
        l.check()
    for rnd in range(2):
        for i in range(2):
            assert torch.equal(outs[("s", rnd, i)], outs[("p", rnd, i)]), (rnd, i)
    for i in range(2):
        assert torch.equal(shared[i].get_fast_weight(), private[i].get_fast_weight())
    o_ref, w_ref = _oracle(cfgs[0])
    assert _rel(_host(outs[("s", 0, 0)]), o_ref) < TOL_BF16


def test_state_persists_across_calls_and_reset():
    """Two calls (the second continues the document) equal the oracle run from
    the first call's final state; reset() restores W_0 exactly."""
    cfg = _bf16_cfg(T=1024, C=128)
    layer, dt = _make_gpu_layer(cfg)
    x = _dev(cfg["x"], dt)
    o1 = layer.forward(x[:512], doc_starts=(0,))
    o2 = layer.forward(x[512:], doc_starts=())
    w = layer.get_fast_weight()
    layer.check()
    o_ref1, w_ref1 = _oracle(cfg, x=cfg["x"][:512], doc_starts=(0,))
    o_ref2, w_ref2 = _oracle(cfg, x=cfg["x"][512:], doc_starts=(), w_init=w_ref1)
    assert _rel(_host(o1), o_ref1) < TOL_BF16
    assert _rel(_host(o2), o_ref2) < TOL_BF16
    assert _rel(_host(w), w_ref2) < TOL_BF16
    layer.reset()
    assert np.array_equal(_host(layer.get_fast_weight()), np.float64(cfg["w_down0"]))


@pytest.mark.parametrize("path", ["tcgen05", "simt"])
def test_fast_weight_round_trip_is_exact(path):
    """set_fast_weight then get_fast_weight gives back every fp32 bit pattern,
    on the tcgen05 path (where the state is kept as a hi and a lo 16-bit
    plane) as on the fp32 one: ordinary values, both signs, values whose low
    16 bits are exactly half way (0x8000) or just below, subnormals, zero."""
    cfg = _bf16_cfg(d=256, f=512, T=64, C=64)
    if path == "simt":
        os.environ["TTT_FORCE_SIMT"] = "1"
    try:
        layer, _ = _make_gpu_layer(cfg)
    finally:
        os.environ.pop("TTT_FORCE_SIMT", None)
    assert layer.path == path
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=(256, 512), dtype=np.uint64).astype(np.uint32)
    bits &= np.uint32(0xBFFFFFFF)                     # finite: exponent below all-ones
    bits[0, :64] = (bits[0, :64] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    bits[1, :64] = (bits[1, :64] & np.uint32(0xFFFF0000)) | np.uint32(0x7FFF)
    bits[2, :64] = bits[2, :64] & np.uint32(0x807FFFFF)  # subnormals
    bits[3, :8] = np.array([0, 0x80000000, 0x00008000, 0x80008000, 0x3F808000, 0xBF808000,
                            0x7F7FFFFF, 0xFF7F7FFF], dtype=np.uint32)
    w = torch.from_numpy(bits.view(np.float32)).cuda()
    layer.set_fast_weight(w)
    back = layer.get_fast_weight()
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy().view(np.uint32), bits)


def test_set_fast_weight_then_continue():
    cfg = _bf16_cfg(T=512, C=64)
    layer, dt = _make_gpu_layer(cfg)
    rng = np.random.default_rng(5)
    w_init = (np.float64(cfg["w_down0"]) + 0.01 * rng.standard_normal(cfg["w_down0"].shape))
    layer.set_fast_weight(torch.from_numpy(w_init.astype(np.float32)).cuda())
    o = layer.forward(_dev(cfg["x"], dt), doc_starts=())
    w = layer.get_fast_weight()
    o_ref, w_ref = _oracle(cfg, doc_starts=(), w_init=w_init.astype(np.float32))
    assert _rel(_host(o), o_ref) < TOL_BF16 and _rel(_host(w), w_ref) < TOL_BF16


def test_batch_slots_are_independent():
    """Per-document fast weights: slot b equals document b run alone."""
    cfgs = [make_layer(256, 512, 640, 64, 5, 0.05, dtype="bf16", seed=0, init="qwen",
                       x_seed=1000 + b) for b in range(3)]
    layer, dt = _make_gpu_layer(cfgs[0], n_docs=3)
    outs = [layer.forward(_dev(c["x"], dt), doc=b) for b, c in enumerate(cfgs)]
    for b, c in enumerate(cfgs):
        o_ref, w_ref = _oracle(c)
        assert _rel(_host(outs[b]), o_ref) < TOL_BF16
        assert _rel(_host(layer.get_fast_weight(b)), w_ref) < TOL_BF16


def test_host_buffer_entry_point():
    cfg = _bf16_cfg(T=512, C=64)
    layer, dt = _make_gpu_layer(cfg)
    xh = _dev(cfg["x"], dt).cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, out_host=oh, doc_starts=(0,))
    torch.cuda.synchronize()
    o_ref, _ = _oracle(cfg)
    assert _rel(_host(oh), o_ref) < TOL_BF16


def test_host_buffer_segments_equal_device_call():
    """A host-buffer call cut into five segments at group starts (4096, 8192,
    13096 and 19049, the last segment being the call's last group alone; the
    call has documents starting at 2048, 9000 and 17001, off the cuts), with
    an X0 that differs from X, equals the device-buffer call bit for bit,
    output and final state."""
    cfg = make_layer(256, 512, 20000, 64, 4, 0.5, dtype="bf16", seed=5, init="qwen",
                     doc_starts=(0, 2048, 9000, 17001))
    dt = torch.bfloat16
    x = _dev(cfg["x"], dt)
    x0 = (x.float() * 0.5 + 0.01).to(dt)
    dev_layer, _ = _make_gpu_layer(cfg)
    o_dev = dev_layer.forward(x, x0, doc_starts=cfg["doc_starts"])
    w_dev = dev_layer.get_fast_weight()
    dev_layer.check()
    host_layer, _ = _make_gpu_layer(cfg)
    xh, x0h = x.cpu().pin_memory(), x0.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    host_layer.forward_host(xh, x0h, out_host=oh, doc_starts=cfg["doc_starts"])
    host_layer.check()
    assert torch.equal(oh, o_dev.cpu())
    assert torch.equal(host_layer.get_fast_weight(), w_dev)


def test_back_to_back_host_calls_with_prefetched_inputs():
    """Four host-buffer calls in a row without synchronising, on different
    documents (a handle that owns its scratch lets each call's input copies
    overlap the previous call's layers, alternating two staging buffers), the
    second and fourth continuing the state of the call before: every output
    and the final state equal the device-buffer calls bit for bit.  A handle
    on a shared scratch (no overlap of input copies) gives the same bits."""
    from chunk_wise_weight_ttt_b300 import TTTMLP, workspace_bytes
    cfg = make_layer(256, 512, 9000, 64, 4, 0.5, dtype="bf16", seed=8, init="qwen")
    dt = torch.bfloat16
    xs = [_dev(cfg["x"], dt)]
    for k in range(1, 4):
        xs.append((xs[0].float() * (1.0 - 0.2 * k) + 0.01 * k).to(dt))
    starts = [(0,), (), (0, 4000), ()]
    dev_layer, _ = _make_gpu_layer(cfg)
    o_dev = [dev_layer.forward(x, doc_starts=ds) for x, ds in zip(xs, starts)]
    w_dev = dev_layer.get_fast_weight()
    dev_layer.check()
    ws = [_dev(cfg[k], dt) for k in ("w_gate", "w_up", "w_down0", "conv_w", "w_target")]
    scratch = torch.empty(workspace_bytes(256, 512, chunk=64, conv_k=4, max_tokens=9000,
                                          part="scratch"), dtype=torch.uint8, device="cuda")
    for layer in (TTTMLP(*ws, chunk=64, eta=cfg["eta"], max_tokens=9000),
                  TTTMLP(*ws, chunk=64, eta=cfg["eta"], max_tokens=9000, scratch=scratch)):
        xh = [x.cpu().pin_memory() for x in xs]
        oh = [torch.empty_like(h).pin_memory() for h in xh]
        for h, o, ds in zip(xh, oh, starts):
            layer.forward_host(h, out_host=o, doc_starts=ds)
        layer.check()
        for k in range(4):
            assert torch.equal(oh[k], o_dev[k].cpu()), k
        assert torch.equal(layer.get_fast_weight(), w_dev)


def test_bad_call_arguments_change_nothing():
    from chunk_wise_weight_ttt_b300 import TTTError
    cfg = _bf16_cfg(T=256, C=64)
    layer, dt = _make_gpu_layer(cfg)
    x = _dev(cfg["x"], dt)
    w_before = layer.get_fast_weight().clone()
    with pytest.raises(TTTError, match="EINVAL"):
        layer.forward(x, doc_starts=(0, 5, 5))          # not strictly increasing
    with pytest.raises(TTTError, match="EINVAL"):
        layer.forward(x, doc_starts=(0, 256))           # out of range
    with pytest.raises(TTTError, match="EINVAL"):
        layer.forward(x, doc=3)                         # no such slot
    with pytest.raises(TTTError, match="EINVAL"):
        layer.forward(x, out=x)                         # output overlaps input
    assert torch.equal(layer.get_fast_weight(), w_before)
    layer.check()


def test_fault_injection_leaves_handle_usable(monkeypatch):
    from chunk_wise_weight_ttt_b300 import TTTError
    cfg = _bf16_cfg(T=256, C=64)
    layer, dt = _make_gpu_layer(cfg)
    x = _dev(cfg["x"], dt)
    monkeypatch.setenv("TTT_FAULT", "forward")
    with pytest.raises(TTTError, match="FAULT_INJECTED"):
        layer.forward(x)
    monkeypatch.delenv("TTT_FAULT")
    o = layer.forward(x)
    o_ref, _ = _oracle(cfg)
    assert _rel(_host(o), o_ref) < TOL_BF16


@pytest.mark.parametrize("hook,T", [("kernel_wait", 512), ("group_wait", 4096)])
def test_bounded_wait_runs_out_and_handle_recovers(monkeypatch, hook, T):
    """TTT_FAULT=kernel_wait makes the target-projection kernel withhold one of
    its own operand loads, TTT_FAULT=group_wait the fused apply+update kernel
    (a launch of two chained groups here, so tiles of the second group wait on
    the withheld tile's completion counter too): the barrier that waits for
    the load never completes, the kernel's bounded waits run out (no GPU
    fault, no hang), ttt_mlp_check reports TTT_ETIMEOUT, and after a reset the
    handle computes correctly."""
    import time
    from chunk_wise_weight_ttt_b300 import TTTError
    cfg = _bf16_cfg(T=T, C=64)
    layer, dt = _make_gpu_layer(cfg)
    x = _dev(cfg["x"], dt)
    layer.check()
    monkeypatch.setenv("TTT_FAULT", hook)
    t0 = time.time()
    layer.forward(x)  # enqueued: the failure is asynchronous
    monkeypatch.delenv("TTT_FAULT")
    with pytest.raises(TTTError, match="ETIMEOUT"):
        layer.check()
    elapsed = time.time() - t0
    print(f"bounded waits ran out after {elapsed:.1f} s")
    assert 1.0 < elapsed < 60.0
    layer.check()  # the error word was cleared
    layer.reset()
    o = layer.forward(x)
    o_ref, _ = _oracle(cfg)
    assert _rel(_host(o), o_ref) < TOL_BF16
    layer.check()


def test_rmsnorm_and_residual_glue():
    from chunk_wise_weight_ttt_b300 import residual_add, rmsnorm
    rng = np.random.default_rng(0)
    h = rng.standard_normal((37, 256)).astype(np.float32) * 3
    ht = torch.from_numpy(h).cuda()
    x = torch.empty((37, 256), dtype=torch.bfloat16, device="cuda")
    rmsnorm(ht, x, 1e-6)
    ref = orc.rms_norm(h, 1e-6)
    assert _rel(_host(x), ref) < 4e-3
    o = torch.from_numpy(rng.standard_normal((37, 256)).astype(np.float32)).cuda()
    residual_add(ht, o)
    assert np.allclose(_host(ht), np.float64(h) + _host(o), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("d,o_dt,x_dt", [(2560, torch.bfloat16, torch.bfloat16), (300, torch.float32, torch.float32),
                                         (256, torch.bfloat16, torch.float32)])
def test_residual_rmsnorm_equals_the_two_glue_calls(d, o_dt, x_dt):
    """The fused residual add + next RMSNorm gives the same bits as the two
    calls one after the other, and RMSNorm of h + o against the oracle."""
    from chunk_wise_weight_ttt_b300 import residual_add, residual_rmsnorm, rmsnorm
    rng = np.random.default_rng(d)
    h = torch.from_numpy(rng.standard_normal((53, d)).astype(np.float32) * 2).cuda()
    o = torch.from_numpy(rng.standard_normal((53, d)).astype(np.float32)).cuda().to(o_dt)
    h1, h2 = h.clone(), h.clone()
    x1 = torch.empty((53, d), dtype=x_dt, device="cuda")
    x2 = torch.empty_like(x1)
    residual_rmsnorm(h1, o, x1, 1e-6)
    residual_add(h2, o)
    rmsnorm(h2, x2, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(h1, h2) and torch.equal(x1, x2)
    ref = orc.rms_norm(_host(h) + _host(o), 1e-6)
    assert _rel(_host(x1), ref) < (4e-3 if x_dt == torch.bfloat16 else 1e-6)
