"""The allocation-free target call (ttt_target_noalloc) against the target the
handle-based forward call computes.

ttt_target_noalloc serves callers that may not allocate device memory (code
running inside another runtime's memory pool, or hosts without cudaMalloc):
its scratch is a fixed file-scope device array instead of a caller workspace.
This file is collected last on purpose; it must pass both on its own in a
fresh process and after every other test, and it runs the call twice in a
row because every call shares (and re-clears) the same scratch array.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from ttt_inputs import make_layer

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2  # the bf16-path tolerance of the parity tests


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to("cuda", torch.bfloat16)


def _p(t):
    return C.c_void_p(t.data_ptr())


def test_target_noalloc_matches_forward_target_twice():
    from chunk_wise_weight_ttt_b300 import TTTMLP, _abi
    lib = _abi.load()
    starts = (0, 377)
    cfg = make_layer(256, 512, 1000, 100, 5, 0.5, dtype="bf16", seed=7, init="qwen",
                     doc_starts=starts)
    T, d = cfg["T"], cfg["d"]
    w = {k: _dev(cfg[k]) for k in ("w_gate", "w_up", "w_down0", "conv_w", "w_target")}
    layer = TTTMLP(w["w_gate"], w["w_up"], w["w_down0"], w["conv_w"], w["w_target"],
                   chunk=cfg["chunk"], eta=cfg["eta"], max_tokens=T)
    x = _dev(cfg["x"])
    layer.forward(x, doc_starts=starts)
    layer.check()
    v_ref = layer.intermediates(T)[1].float().clone()

    arr = (C.c_int64 * len(starts))(*starts)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    v = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    for call in range(2):
        v.fill_(float("nan"))
        st = lib.ttt_target_noalloc(_p(x), _p(w["conv_w"]), _p(w["w_target"]), T, d,
                                    cfg["k"], cfg["chunk"], arr, len(starts), cfg["eta"], _p(v),
                                    _p(status), stream)
        assert st == _abi.TTT_OK, lib.ttt_mlp_last_error(None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        err = float(torch.linalg.norm(v.float() - v_ref) / torch.linalg.norm(v_ref))
        print(f"call {call}: rel err vs forward-call target {err:.3e}")
        assert err <= TOL_BF16


def test_target_noalloc_rejects_oversize():
    from chunk_wise_weight_ttt_b300 import _abi
    lib = _abi.load()
    d = 2560
    n = (_abi.NOALLOC_SCRATCH_BYTES - 2 * d * d) // (2 * d) + 1  # one token too many
    fake = C.c_void_p(0x1000)  # never dereferenced: the size check comes first
    st = lib.ttt_target_noalloc(fake, fake, fake, n, d, 5, 256, None, 0, 1e-3, fake, None, None)
    assert st == _abi.TTT_EUNSUPPORTED
    assert b"scratch" in lib.ttt_mlp_last_error(None)
