"""PyTorch-facing binding of the TTT-MLP layer (argument marshalling only).

PyTorch supplies device memory (weights, workspace, activations) and the CUDA
stream; every computation runs in libttt_mlp.so's kernels.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Sequence

import torch

from . import _abi
from ._abi import Config, TTTError, TTT_BF16, TTT_F32

_DT = {torch.float32: TTT_F32, torch.bfloat16: TTT_BF16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check(lib, h, status: int):
    if status != _abi.TTT_OK:
        msg = lib.ttt_mlp_last_error(h).decode(errors="replace")
        raise TTTError(status, msg)


def _doc_array(doc_starts: Optional[Sequence[int]]):
    if not doc_starts:
        return None, 0
    arr = (C.c_int64 * len(doc_starts))(*[int(s) for s in doc_starts])
    return arr, len(doc_starts)


class TTTMLP:
    """One SwiGLU MLP block whose down projection is an In-Place TTT fast weight.

    Weights are CUDA tensors in nn.Linear layouts (w_gate, w_up: f x d;
    w_down0: d x f) plus conv_w (k x d) and w_target (d x d, in x out).  The
    object keeps references to the weights and owns its workspace tensor, or
    borrows `workspace` (a uint8 CUDA tensor of at least workspace_bytes())
    when one is given.
    """

    def __init__(self, w_gate, w_up, w_down0, conv_w, w_target, *, chunk: int, eta: float,
                 n_docs: int = 1, max_tokens: int, stream=None, workspace=None, scratch=None,
                 target_mode: int = _abi.TTT_TARGET_NEXT, clip_tau: float = 0.0):
        self.lib = _abi.load()
        dt = w_gate.dtype
        if dt not in _DT:
            raise TypeError("weights must be float32 or bfloat16")
        ws = [w_gate, w_up, w_down0, conv_w, w_target]
        if any((not t.is_cuda) or t.dtype != dt or not t.is_contiguous() for t in ws):
            raise ValueError("weights must be contiguous CUDA tensors of one dtype")
        f, d = w_gate.shape
        self.d, self.f, self.k = d, f, conv_w.shape[0]
        self.dtype = dt
        self.cfg = Config(d=d, f=f, chunk=chunk, conv_k=self.k, n_docs=n_docs, eta=eta,
                          act_dtype=_DT[dt], max_tokens=max_tokens, target_mode=target_mode,
                          clip_tau=clip_tau or 0.0)
        cfg = C.byref(self.cfg)
        self._weights = ws
        h = C.c_void_p()
        if scratch is None:
            nbytes = self.lib.ttt_mlp_workspace_bytes(cfg)
            if nbytes == 0:
                raise TTTError(_abi.TTT_EINVAL, "invalid configuration")
            if workspace is None:
                workspace = torch.empty(nbytes, dtype=torch.uint8, device=w_gate.device)
            elif workspace.dtype != torch.uint8 or workspace.numel() < nbytes or not workspace.is_cuda:
                raise ValueError(f"workspace must be a CUDA uint8 tensor of at least {nbytes} bytes")
            self.workspace = workspace
            st = self.lib.ttt_mlp_create(cfg, *[_ptr(t) for t in ws], _ptr(self.workspace), nbytes,
                                         _stream(stream), C.byref(h))
        else:
            # own state, scratch shared with other handles whose calls are ordered
            sbytes = self.lib.ttt_mlp_state_bytes(cfg)
            xbytes = self.lib.ttt_mlp_scratch_bytes(cfg)
            if sbytes == 0:
                raise TTTError(_abi.TTT_EINVAL, "invalid configuration")
            if scratch.dtype != torch.uint8 or scratch.numel() < xbytes or not scratch.is_cuda:
                raise ValueError(f"scratch must be a CUDA uint8 tensor of at least {xbytes} bytes")
            self.state = torch.empty(sbytes, dtype=torch.uint8, device=w_gate.device)
            self.workspace = scratch
            st = self.lib.ttt_mlp_create_split(cfg, *[_ptr(t) for t in ws], _ptr(self.state), sbytes,
                                               _ptr(scratch), scratch.numel(), _stream(stream),
                                               C.byref(h))
        _check(self.lib, None, st)
        self.h = h

    @property
    def path(self) -> str:
        return self.lib.ttt_mlp_path(self.h).decode()

    def forward(self, x: torch.Tensor, x0: Optional[torch.Tensor] = None, *, doc: int = 0,
                doc_starts: Optional[Sequence[int]] = (0,), out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
        """O for the tokens of x (n x d), continuing slot `doc`'s fast weight;
        `doc_starts` are offsets where a document begins (W reset to W_0)."""
        x0 = x if x0 is None else x0
        if out is None:
            out = torch.empty_like(x)
        arr, nds = _doc_array(doc_starts)
        st = self.lib.ttt_mlp_forward_chunks(self.h, doc, _ptr(x), _ptr(x0), x.shape[0], arr, nds,
                                             _ptr(out), _stream(stream))
        _check(self.lib, self.h, st)
        return out

    __call__ = forward

    def forward_static(self, x: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
        """The block's static MLP, SwiGLU(x) W_0^T (no fast weight)."""
        if out is None:
            out = torch.empty_like(x)
        st = self.lib.ttt_mlp_forward_static(self.h, _ptr(x), x.shape[0], _ptr(out), _stream(stream))
        _check(self.lib, self.h, st)
        return out

    def forward_host(self, x_host: torch.Tensor, x0_host: Optional[torch.Tensor] = None, *,
                     doc: int = 0, doc_starts: Optional[Sequence[int]] = (0,),
                     out_host: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """Same as forward() with host tensors (pinned for asynchronous copies);
        the copies run on the stream, so synchronise before reading the result."""
        x0_host = x_host if x0_host is None else x0_host
        if out_host is None:
            out_host = torch.empty_like(x_host)
        arr, nds = _doc_array(doc_starts)
        st = self.lib.ttt_mlp_forward_chunks_host(self.h, doc, _ptr(x_host), _ptr(x0_host),
                                                  x_host.shape[0], arr, nds, _ptr(out_host),
                                                  _stream(stream))
        _check(self.lib, self.h, st)
        return out_host

    def intermediates(self, n_tokens: int):
        """(Z, V) of the last forward call as tensor views into the workspace."""
        z, v, dt = C.c_void_p(), C.c_void_p(), C.c_int32()
        _check(self.lib, self.h, self.lib.ttt_mlp_intermediates(self.h, C.byref(z), C.byref(v),
                                                                C.byref(dt)))
        tdt = torch.bfloat16 if dt.value == TTT_BF16 else torch.float32
        esz = 2 if dt.value == TTT_BF16 else 4
        base = self.workspace.data_ptr()
        zt = self.workspace[z.value - base: z.value - base + n_tokens * self.f * esz]
        vt = self.workspace[v.value - base: v.value - base + n_tokens * self.d * esz]
        return (zt.view(tdt).view(n_tokens, self.f), vt.view(tdt).view(n_tokens, self.d))

    def reset(self, doc: int = -1, stream=None):
        _check(self.lib, self.h, self.lib.ttt_mlp_reset(self.h, doc, _stream(stream)))

    def get_fast_weight(self, doc: int = 0, stream=None) -> torch.Tensor:
        w = torch.empty((self.d, self.f), dtype=torch.float32, device=self.workspace.device)
        _check(self.lib, self.h, self.lib.ttt_mlp_get_fast_weight(self.h, doc, _ptr(w),
                                                                  _stream(stream)))
        return w

    def set_fast_weight(self, w: torch.Tensor, doc: int = 0, stream=None):
        if w.dtype != torch.float32 or tuple(w.shape) != (self.d, self.f) or not w.is_contiguous():
            raise ValueError("fast weight must be a contiguous float32 d x f tensor")
        _check(self.lib, self.h, self.lib.ttt_mlp_set_fast_weight(self.h, doc, _ptr(w),
                                                                  _stream(stream)))

    def profile(self, enable: bool = True):
        """Start (clearing earlier records) or stop recording phase events."""
        _check(self.lib, self.h, self.lib.ttt_mlp_profile_enable(self.h, 1 if enable else 0))

    def profile_read(self) -> dict:
        """Per-phase milliseconds summed over the profiled calls, and counts."""
        ms = (C.c_float * 5)()
        cnt = (C.c_int64 * 3)()
        _check(self.lib, self.h, self.lib.ttt_mlp_profile_read(self.h, ms, cnt))
        names = ("conv", "swiglu", "vproj", "gram", "group")
        return {"ms": dict(zip(names, list(ms))), "calls": cnt[0], "group_launches": cnt[1],
                "launches": cnt[2]}

    def check(self, stream=None):
        _check(self.lib, self.h, self.lib.ttt_mlp_check(self.h, _stream(stream)))

    def close(self):
        if getattr(self, "h", None):
            self.lib.ttt_mlp_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def workspace_bytes(d: int, f: int, *, chunk: int, conv_k: int, dtype=torch.bfloat16,
                    n_docs: int = 1, max_tokens: int, eta: float = 0.0,
                    target_mode: int = _abi.TTT_TARGET_NEXT, clip_tau: float = 0.0,
                    part: str = "all") -> int:
    """Device workspace (bytes) a layer of this shape needs: the whole
    workspace (part="all"), or its per-handle state or shareable scratch part."""
    lib = _abi.load()
    cfg = Config(d=d, f=f, chunk=chunk, conv_k=conv_k, n_docs=n_docs, eta=eta, act_dtype=_DT[dtype],
                 max_tokens=max_tokens, target_mode=target_mode, clip_tau=clip_tau or 0.0)
    fn = {"all": lib.ttt_mlp_workspace_bytes, "state": lib.ttt_mlp_state_bytes,
          "scratch": lib.ttt_mlp_scratch_bytes}[part]
    return int(fn(C.byref(cfg)))


def is_ttt_layer(layer: int, ttt_every: int) -> bool:
    """Whether 0-based block `layer` carries In-Place TTT when every
    `ttt_every`-th block does: the ttt_every-th, 2*ttt_every-th, ... blocks
    (1-based), so ttt_every=1 makes every block a TTT block."""
    return (layer + 1) % ttt_every == 0


class TTTStack:
    """Pre-norm residual stack of SwiGLU MLP blocks (no attention):
        h_{l+1} = h_l + MLP_l(RMSNorm(h_l)),   X0 = h_0 for every TTT block,
    where MLP_l is an In-Place TTT block (fast W_down) when
    is_ttt_layer(l, ttt_every) and the static SwiGLU MLP otherwise.
    Layer-major: each block runs its chunk recursion over the whole call before
    the next block starts (the recursion is per block and nothing else mixes
    tokens).  Every block has its own handle, made once: its fast-weight state
    is its own and the per-call scratch is shared (the blocks run one after
    another on one stream).  A call processes whole documents: the fast
    weights start at W_0 (doc_starts must contain 0).

    layers: list of dicts with CUDA tensors w_gate, w_up, w_down0, conv_w,
    w_target (one dtype).  h is fp32 (T x d); activations are cast to the
    weights' dtype.
    """

    def __init__(self, layers, *, chunk: int, eta: float, max_tokens: int, eps: float = 1e-6,
                 target_mode: int = _abi.TTT_TARGET_NEXT, clip_tau: float = 0.0,
                 ttt_every: int = 1, stream=None):
        if ttt_every < 1:
            raise ValueError("ttt_every must be >= 1")
        self.layers = layers
        w = layers[0]
        self.dtype = w["w_gate"].dtype
        f, d = w["w_gate"].shape
        self.d, self.f, self.k = d, f, w["conv_w"].shape[0]
        self.chunk, self.eta, self.max_tokens, self.eps = chunk, eta, max_tokens, eps
        self.target_mode, self.clip_tau, self.ttt_every = target_mode, clip_tau, ttt_every
        nbytes = workspace_bytes(d, f, chunk=chunk, conv_k=self.k, dtype=self.dtype,
                                 max_tokens=max_tokens, eta=eta, target_mode=target_mode,
                                 clip_tau=clip_tau, part="scratch")
        self.scratch = torch.empty(nbytes, dtype=torch.uint8, device=w["w_gate"].device)
        self.blocks = [TTTMLP(lw["w_gate"], lw["w_up"], lw["w_down0"], lw["conv_w"], lw["w_target"],
                              chunk=chunk, eta=eta, max_tokens=max_tokens, stream=stream,
                              scratch=self.scratch, target_mode=target_mode, clip_tau=clip_tau)
                       for lw in layers]

    def forward(self, h0: torch.Tensor, doc_starts: Sequence[int] = (0,), stream=None,
                n_layers: Optional[int] = None) -> torch.Tensor:
        if not doc_starts or int(doc_starts[0]) != 0:
            raise ValueError("a stack call processes whole documents: doc_starts must start with 0")
        if h0.dtype != torch.float32 or h0.dim() != 2 or h0.shape[1] != self.d:
            raise ValueError("h0 must be a float32 (T x d) CUDA tensor")
        h = h0.clone()
        x0 = h0.to(self.dtype)
        x = torch.empty(h0.shape, dtype=self.dtype, device=h0.device)
        o = torch.empty_like(x)
        n = n_layers or len(self.blocks)
        rmsnorm(h, x, self.eps, stream=stream)
        for li, blk in enumerate(self.blocks[:n]):
            if is_ttt_layer(li, self.ttt_every):
                blk.forward(x, x0, doc_starts=doc_starts, out=o, stream=stream)
            else:
                blk.forward_static(x, out=o, stream=stream)
            if li + 1 < n:
                residual_rmsnorm(h, o, x, self.eps, stream=stream)  # and the next block's input
            else:
                residual_add(h, o, stream=stream)
        return h

    __call__ = forward

    def check(self, stream=None):
        """Synchronise and raise if any block's in-kernel wait ran out."""
        for blk in self.blocks:
            blk.check(stream=stream)

    def close(self):
        for blk in self.blocks:
            blk.close()


def rmsnorm(h: torch.Tensor, out: torch.Tensor, eps: float = 1e-6, stream=None) -> torch.Tensor:
    lib = _abi.load()
    st = lib.ttt_rmsnorm(_ptr(h), _ptr(out), h.shape[0], h.shape[1], eps, _DT[out.dtype],
                         _stream(stream))
    _check(lib, None, st)
    return out


def residual_rmsnorm(h: torch.Tensor, o: torch.Tensor, out: torch.Tensor, eps: float = 1e-6,
                     stream=None) -> torch.Tensor:
    """h += o, then out = RMSNorm(h), in one pass over h."""
    lib = _abi.load()
    st = lib.ttt_residual_rmsnorm(_ptr(h), _ptr(o), _ptr(out), h.shape[0], h.shape[1], eps,
                                  _DT[o.dtype], _DT[out.dtype], _stream(stream))
    _check(lib, None, st)
    return out


def residual_add(h: torch.Tensor, o: torch.Tensor, stream=None) -> torch.Tensor:
    lib = _abi.load()
    st = lib.ttt_residual_add(_ptr(h), _ptr(o), h.shape[0], h.shape[1], _DT[o.dtype],
                              _stream(stream))
    _check(lib, None, st)
    return h
