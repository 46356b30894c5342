"""The allocation-free target call (ttt_target_noalloc).

ttt_target_noalloc serves callers that may not allocate device memory (code
running inside another runtime's memory pool, or hosts without cudaMalloc):
its scratch is a fixed file-scope device array instead of a caller workspace.
Its target V = eta * Conv1D(X0) W_target is checked against the CPU oracle
(chunk by chunk, chunking restarted at document starts off the chunk grid) and
bit for bit against the target the handle-based forward call computes with
the same kernels.  This file is collected last on purpose; it must pass both
on its own in a fresh process and after every other test, and it runs the call
twice in a row because every call shares (and re-clears) the same scratch.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle.ttt_oracle as orc
from ttt_inputs import make_layer

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2  # the bf16-path tolerance of the parity tests


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to("cuda", torch.bfloat16)


def _p(t):
    return C.c_void_p(t.data_ptr())


def _oracle_target(cfg, starts):
    """eta * Conv1D(X0) W_target with the chunking of a call that has these
    document starts (the oracle's chunk spans)."""
    v = np.zeros((cfg["T"], cfg["d"]))
    for s, e, _ in orc.chunk_spans(cfg["T"], cfg["chunk"], starts):
        v[s:e] = cfg["eta"] * orc.chunk_target(cfg["x0"][s:e], cfg["conv_w"], cfg["w_target"])
    return v


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _noalloc(lib, x, w, cfg, starts, v, status):
    arr = (C.c_int64 * len(starts))(*starts) if starts else None
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ttt_target_noalloc(_p(x), _p(w["conv_w"]), _p(w["w_target"]), cfg["T"], cfg["d"],
                                  cfg["k"], cfg["chunk"], arr, len(starts), cfg["eta"], _p(v),
                                  None if status is None else _p(status), stream)


def test_target_noalloc_matches_oracle_and_forward_target_twice():
    from chunk_wise_weight_ttt_b300 import TTTMLP, _abi
    lib = _abi.load()
    starts = (0, 377, 640)  # documents starting off the 100-token chunk grid
    cfg = make_layer(256, 512, 1000, 100, 5, 0.5, dtype="bf16", seed=7, init="qwen",
                     doc_starts=starts)
    T, d = cfg["T"], cfg["d"]
    w = {k: _dev(cfg[k]) for k in ("w_gate", "w_up", "w_down0", "conv_w", "w_target")}
    layer = TTTMLP(w["w_gate"], w["w_up"], w["w_down0"], w["conv_w"], w["w_target"],
                   chunk=cfg["chunk"], eta=cfg["eta"], max_tokens=T)
    x = _dev(cfg["x"])
    layer.forward(x, doc_starts=starts)
    layer.check()
    v_fwd = layer.intermediates(T)[1].clone()
    v_ref = _oracle_target(cfg, starts)

    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    v = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    for call in range(2):
        v.fill_(float("nan"))
        st = _noalloc(lib, x, w, cfg, starts, v, status)
        assert st == _abi.TTT_OK, lib.ttt_mlp_last_error(None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        err = _rel(v.double().cpu().numpy(), v_ref)
        print(f"call {call}: rel err vs oracle target {err:.3e}; "
              f"bitwise equal to the forward call's target: {torch.equal(v, v_fwd)}")
        assert err <= TOL_BF16
        assert torch.equal(v, v_fwd)


def test_target_noalloc_at_the_exact_scratch_size():
    """The largest call that fits the fixed array (2*d*d + 2*n*d + 512 bytes ==
    TTT_NOALLOC_SCRATCH_BYTES at d=256) runs and matches the oracle; one token
    more is refused before anything is enqueued."""
    from chunk_wise_weight_ttt_b300 import _abi
    lib = _abi.load()
    d = 256
    n = (_abi.NOALLOC_SCRATCH_BYTES - 2 * d * d - 512) // (2 * d)
    assert 2 * d * d + 2 * n * d + 512 == _abi.NOALLOC_SCRATCH_BYTES
    cfg = make_layer(d, 256, n, 256, 5, 1e-3, dtype="bf16", seed=9, init="qwen")
    w = {k: _dev(cfg[k]) for k in ("conv_w", "w_target")}
    x = _dev(cfg["x"])
    v = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    st = _noalloc(lib, x, w, cfg, (0,), v, status)
    assert st == _abi.TTT_OK, lib.ttt_mlp_last_error(None)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    err = _rel(v.double().cpu().numpy(), _oracle_target(cfg, (0,)))
    print(f"exact-fit call ({n} tokens): rel err vs oracle target {err:.3e}")
    assert err <= TOL_BF16
    bigger = dict(cfg, T=n + 1)
    st = _noalloc(lib, x, w, bigger, (0,), v, None)
    assert st == _abi.TTT_EUNSUPPORTED
    assert b"scratch" in lib.ttt_mlp_last_error(None)


def test_target_noalloc_rejects_oversize():
    from chunk_wise_weight_ttt_b300 import _abi
    lib = _abi.load()
    d = 2560
    n = (_abi.NOALLOC_SCRATCH_BYTES - 2 * d * d) // (2 * d) + 1  # one token too many
    fake = C.c_void_p(0x1000)  # never dereferenced: the size check comes first
    st = lib.ttt_target_noalloc(fake, fake, fake, n, d, 5, 256, None, 0, 1e-3, fake, None, None)
    assert st == _abi.TTT_EUNSUPPORTED
    assert b"scratch" in lib.ttt_mlp_last_error(None)
