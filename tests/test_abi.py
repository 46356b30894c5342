"""Host-side checks of the C ABI: the library loads, exports every function the
header declares, validates configurations and arguments before touching CUDA,
and honours the host-side fault-injection hook.  No kernel runs here."""
import ctypes as C
import os
import re

import pytest

from chunk_wise_weight_ttt_b300 import _abi
from chunk_wise_weight_ttt_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ttt_mlp.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _abi.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ttt_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    declared = _declared_functions()
    assert declared, "no functions parsed from the header"
    assert sorted(_abi.SIGNATURES) == declared


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def _cfg(**kw):
    c = dict(d=64, f=256, chunk=64, conv_k=4, n_docs=1, eta=0.01, act_dtype=_abi.TTT_F32,
             max_tokens=1024)
    c.update(kw)
    return _abi.Config(**c)


def test_workspace_bytes_valid_and_invalid(lib):
    good = lib.ttt_mlp_workspace_bytes(C.byref(_cfg()))
    # at least the fp32 fast weight + Z/U/V + staging
    assert good >= 64 * 256 * 4 + 1024 * (256 + 2 * 64) * 4
    for bad in [dict(d=0), dict(d=12), dict(f=7), dict(chunk=0), dict(chunk=1025),
                dict(conv_k=0), dict(conv_k=9), dict(n_docs=0), dict(act_dtype=7),
                dict(max_tokens=0), dict(eta=float("nan")), dict(target_mode=3),
                dict(target_mode=-1), dict(clip_tau=-1.0), dict(clip_tau=float("inf"))]:
        assert lib.ttt_mlp_workspace_bytes(C.byref(_cfg(**bad))) == 0, bad
    assert lib.ttt_mlp_workspace_bytes(None) == 0


def test_clipping_adds_gram_workspace(lib):
    plain = lib.ttt_mlp_workspace_bytes(C.byref(_cfg()))
    clip = lib.ttt_mlp_workspace_bytes(C.byref(_cfg(clip_tau=1e-5)))
    assert clip >= plain + 2 * 64 * 64 * 4  # two fp32 same-chunk Gram blocks (fp32 path)
    assert lib.ttt_mlp_workspace_bytes(C.byref(_cfg(target_mode=2))) == plain


def test_workspace_bytes_qwen_layer(lib):
    c = _cfg(d=2560, f=9728, chunk=256, conv_k=5, act_dtype=_abi.TTT_BF16, max_tokens=32768)
    b = lib.ttt_mlp_workspace_bytes(C.byref(c))
    w = 2560 * 9728 * 4
    assert w < b < 8 * 2 ** 30


def test_create_rejects_bad_arguments_without_cuda(lib):
    h = C.c_void_p()
    fake = C.c_void_p(0x1000)  # never dereferenced: validation fails first
    # NULL weight pointer
    st = lib.ttt_mlp_create(C.byref(_cfg()), None, fake, fake, fake, fake, fake, 1 << 30, None,
                            C.byref(h))
    assert st == _abi.TTT_EINVAL and not h.value
    assert b"non-NULL" in lib.ttt_mlp_last_error(None)
    # misaligned weight pointer
    st = lib.ttt_mlp_create(C.byref(_cfg()), C.c_void_p(0x1001), fake, fake, fake, fake, fake,
                            1 << 30, None, C.byref(h))
    assert st == _abi.TTT_EINVAL
    # workspace too small
    st = lib.ttt_mlp_create(C.byref(_cfg()), fake, fake, fake, fake, fake, fake, 16, None,
                            C.byref(h))
    assert st == _abi.TTT_EINVAL
    assert b"workspace" in lib.ttt_mlp_last_error(None)
    # invalid configuration
    st = lib.ttt_mlp_create(C.byref(_cfg(chunk=0)), fake, fake, fake, fake, fake, fake, 1 << 30,
                            None, C.byref(h))
    assert st == _abi.TTT_EINVAL
    # NULL out pointer
    assert lib.ttt_mlp_create(C.byref(_cfg()), fake, fake, fake, fake, fake, fake, 1 << 30, None,
                              None) == _abi.TTT_EINVAL


def test_null_handle_calls_fail_cleanly(lib):
    assert lib.ttt_mlp_forward_chunks(None, 0, None, None, 0, None, 0, None, None) == _abi.TTT_EINVAL
    assert lib.ttt_mlp_reset(None, 0, None) == _abi.TTT_EINVAL
    assert lib.ttt_mlp_get_fast_weight(None, 0, None, None) == _abi.TTT_EINVAL
    assert lib.ttt_mlp_set_fast_weight(None, 0, None, None) == _abi.TTT_EINVAL
    assert lib.ttt_mlp_check(None, None) == _abi.TTT_EINVAL
    assert lib.ttt_mlp_destroy(None) == _abi.TTT_EINVAL
    assert lib.ttt_mlp_path(None) == b"simt"
    assert lib.ttt_rmsnorm(None, None, 4, 0, 1e-6, 0, None) == _abi.TTT_EINVAL
    assert lib.ttt_residual_add(None, None, 4, 8, 3, None) == _abi.TTT_EINVAL


def test_fault_injection_create(lib, monkeypatch):
    monkeypatch.setenv("TTT_FAULT", "create")
    h = C.c_void_p()
    fake = C.c_void_p(0x1000)
    st = lib.ttt_mlp_create(C.byref(_cfg()), fake, fake, fake, fake, fake, fake, 1 << 30, None,
                            C.byref(h))
    assert st == _abi.TTT_EFAULT_INJECTED and not h.value
    assert b"fault injected" in lib.ttt_mlp_last_error(None)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _abi.load(str(tmp_path / "nope.so"))
