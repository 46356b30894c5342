"""CPU fp64 oracle for the In-Place TTT chunk-wise fast-weight (W_down) path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module; only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg do.  It shares no code with the CUDA path: the only common
module is the seeded input generator, which holds none of the method's
arithmetic.

It computes, in float64 on the same bf16/fp32-stored inputs the GPU sees,
exactly what the method defines, step by step in the order the pages give it.
numpy's matmul is the one library primitive used; nothing is blocked, fused or
reordered beyond the definitions.

Sources (titles of the pages; sections as printed on them):
  [SUM]  "In-Place Test-Time Training", paperlayer.ai summary of arXiv
         2604.06169v1 -- sections 3 (In-Place Adaptation, Chunk-Wise Updates,
         LM-Aligned Objective), B (Context Parallel Algorithm), C.2, C.3.
  [BLOG] iplexlaw.co.kr walkthrough of arXiv 2604.06169v1 -- sections 2, 3, 4, 6.

Readings taken where the pages leave a step open (each is repeated in the
design notes):
  R1  The target convolution is a depthwise forward window that starts at the
      next token: U[t] = sum_{j<k} conv[j] * X0[t+1+j], with every term whose
      token lies at or past the end of t's chunk set to zero.  ("future-token
      information", [SUM] 3 LM-Aligned Objective; "next token or a combination
      of nearby future tokens", [BLOG] 4; no pull from other chunks, [BLOG] 6.)
  R2  No bias in the convolution or in W_target (none is mentioned).
  R3  The update is W <- W + eta * V^T Z with no 1/C factor ([BLOG] 2 and 4).
  R4  Chunking restarts at every document start; a document's last chunk may
      be shorter than C.  A call's trailing partial chunk is a short chunk.
  R5  Update clipping ([SUM] C.2; [BLOG] 6) is optional and per chunk: when a
      threshold tau is given, the chunk's delta eta V^T Z is scaled by
      min(1, tau / ||eta V^T Z||_F) before it is added (the pages bound "the
      Frobenius norm of the update delta"; one delta per chunk).
  R6  Target variants (ablation axes of [SUM] 4 and the reconstruction target
      of [SUM] 2 / [BLOG] 4) are windows at other offsets, cut at the chunk
      edges like R1: mode 1 starts at the current token (k = 1 is the
      reconstruction target X0[t]); mode 2 is a causal window that ends at the
      next token.
  R13 Placement ([SUM] C.3 "TTT integration"; [BLOG] 6 and FAQ): with TTT in
      every s-th MLP block, the TTT blocks are the s-th, 2s-th, ... blocks
      counted from 1 (0-based l with (l + 1) % s == 0); every other block is
      the unchanged SwiGLU MLP with its frozen W_down.  s = 1 puts TTT in
      every block.

Function-level parity status: every public function here is pinned by a
"not gpu" test (brute force, closed forms, library routines, invariants).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "TARGET_NEXT",
    "TARGET_CURRENT",
    "TARGET_CAUSAL",
    "silu",
    "swiglu_intermediate",
    "chunk_target_source",
    "chunk_target",
    "clip_delta",
    "chunk_delta_norms",
    "chunk_spans",
    "ttt_layer",
    "ttt_core",
    "ttt_layer_rows",
    "rms_norm",
    "static_mlp",
    "ttt_stack",
]


# Target windows (reading R1 and R6): offset of tap j from token t.
TARGET_NEXT = 0     # X0[t+1+j]
TARGET_CURRENT = 1  # X0[t+j]
TARGET_CAUSAL = 2   # X0[t+1-j]


def _tap_offset(mode: int, j: int) -> int:
    if mode == TARGET_NEXT:
        return 1 + j
    if mode == TARGET_CURRENT:
        return j
    if mode == TARGET_CAUSAL:
        return 1 - j
    raise ValueError(f"unknown target mode {mode}")


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def silu(a: np.ndarray) -> np.ndarray:
    """SiLU(a) = a * sigmoid(a) = a / (1 + exp(-a)).

    SwiGLU activation ([SUM] C.3 "SwiGLU activations")."""
    a = _f64(a)
    return a / (1.0 + np.exp(-a))


def swiglu_intermediate(x, w_gate, w_up) -> np.ndarray:
    """Gated intermediate activation Z = SiLU(X W_gate^T) * (X W_up^T).

    The two projections of the gated MLP are combined into Z; W_gate and W_up
    stay frozen ([BLOG] 2; [SUM] 3 In-Place Adaptation).  x: n x d,
    w_gate/w_up: f x d (nn.Linear layout) -> n x f."""
    x = _f64(x)
    return silu(x @ _f64(w_gate).T) * (x @ _f64(w_up).T)


def chunk_target_source(x0_chunk, conv_w, mode: int = TARGET_NEXT) -> np.ndarray:
    """Depthwise causal-shifted Conv1D of one chunk's embeddings (reading R1).

    U[t] = sum_{j=0}^{k-1} conv[j] (elementwise) X0[t+1+j], terms whose token
    index t+1+j reaches the chunk's end are zero, so no information enters
    from another chunk ([BLOG] 6; "causal padding", [SUM] B).  Other windows
    (reading R6): mode TARGET_CURRENT uses X0[t+j], TARGET_CAUSAL X0[t+1-j];
    every term whose token lies outside the chunk is zero.
    x0_chunk: n x d, conv_w: k x d -> n x d."""
    x0 = _f64(x0_chunk)
    cw = _f64(conv_w)
    n, d = x0.shape
    u = np.zeros((n, d), dtype=np.float64)
    for j in range(cw.shape[0]):
        o = _tap_offset(mode, j)
        t0, t1 = max(0, -o), min(n, n - o)  # tokens t with 0 <= t+o < n
        if t1 > t0:
            u[t0:t1] += cw[j][None, :] * x0[t0 + o:t1 + o]
    return u


def chunk_target(x0_chunk, conv_w, w_target, mode: int = TARGET_NEXT) -> np.ndarray:
    """LM-aligned target V = Conv1D(X0) W_target ([SUM] 3 LM-Aligned Objective;
    [BLOG] 4).  w_target: d x d, given as in x out."""
    return chunk_target_source(x0_chunk, conv_w, mode) @ _f64(w_target)


def clip_delta(delta, clip_tau):
    """Per-chunk update clipping (reading R5): delta * min(1, tau/||delta||_F);
    no clipping when clip_tau is None or 0."""
    if not clip_tau:
        return delta
    nrm = float(np.linalg.norm(delta))
    return delta * (clip_tau / nrm) if nrm > clip_tau else delta


def chunk_spans(n_tokens: int, chunk: int, doc_starts=(0,)):
    """Chunk boundaries of one call: list of (start, end, resets_w).

    Non-overlapping chunks of ``chunk`` tokens processed in order ([SUM] 3
    Chunk-Wise Updates); chunking restarts at each document start, where the
    fast weight is reset ([SUM] B; reading R4).  The call itself starts a fresh
    chunk at token 0 whether or not 0 is a document start."""
    if chunk < 1:
        raise ValueError("chunk must be >= 1")
    starts = sorted(set(int(s) for s in (doc_starts or ())))
    if any(s < 0 or s >= max(n_tokens, 1) for s in starts) and n_tokens > 0:
        raise ValueError("document starts must lie in [0, n_tokens)")
    cuts = [0] + [s for s in starts if s > 0] + [n_tokens]
    spans = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        doc_reset = a in starts
        t = a
        while t < b:
            e = min(t + chunk, b)
            spans.append((t, e, doc_reset and t == a))
            t = e
    return spans


def ttt_layer(x, x0, w_gate, w_up, w_down0, conv_w, w_target, eta, chunk,
              doc_starts=(0,), w_init=None, target_mode=TARGET_NEXT, clip_tau=None):
    """One TTT-MLP layer over one call's tokens, the sequential recursion.

    For every chunk c in order ([BLOG] 3 "apply then update"):
      Z_c = SiLU(X_c W_gate^T) * (X_c W_up^T)
      O_c = Z_c W_c^T                      (the state before this chunk's update)
      V_c = Conv1D(X0_c) W_target          (chunk-local target)
      W_{c+1} = W_c + eta V_c^T Z_c        ([BLOG] 2, 4)
    W starts at ``w_init`` (default W_0 = w_down0) and is reset to W_0 at each
    document start ([SUM] B).  ``target_mode`` picks the target window (R1,
    R6); ``clip_tau`` clips each chunk's delta (R5).  Returns (O n x d, final
    W d x f), float64."""
    x = _f64(x)
    x0 = _f64(x0)
    w0 = _f64(w_down0)
    n = x.shape[0]
    W = w0.copy() if w_init is None else _f64(w_init).copy()
    out = np.zeros((n, w0.shape[0]), dtype=np.float64)
    for s, e, reset in chunk_spans(n, chunk, doc_starts):
        if reset:
            W = w0.copy()
        z = swiglu_intermediate(x[s:e], w_gate, w_up)
        out[s:e] = z @ W.T
        v = chunk_target(x0[s:e], conv_w, w_target, target_mode)
        W = W + clip_delta(float(eta) * (v.T @ z), clip_tau)
    return out, W


def ttt_core(z, v, w_down0, eta, chunk, doc_starts=(0,), w_init=None):
    """The chunk recursion alone, given the per-token intermediates.

    For every chunk c in order ([BLOG] 3 "apply then update"):
      O_c = Z_c W_c^T                      (the state before this chunk's update)
      W_{c+1} = W_c + eta V_c^T Z_c        ([BLOG] 2, 4)
    with W starting at ``w_init`` (default W_0) and reset to W_0 at each
    document start ([SUM] B).  ``z`` (n x f) is the gated intermediate and
    ``v`` (n x d) the target, each row computed for the chunk that holds it
    (the target is chunk-local, reading R1).  This is the apply+update part of
    ttt_layer without the producers; no clipping.  Returns (O n x d, final W)."""
    z = _f64(z)
    v = _f64(v)
    w0 = _f64(w_down0)
    n = z.shape[0]
    W = w0.copy() if w_init is None else _f64(w_init).copy()
    out = np.zeros((n, w0.shape[0]), dtype=np.float64)
    for s, e, reset in chunk_spans(n, chunk, doc_starts):
        if reset:
            W = w0.copy()
        out[s:e] = z[s:e] @ W.T
        W = W + float(eta) * (v[s:e].T @ z[s:e])
    return out, W


def ttt_layer_rows(x, x0, w_gate, w_up, w_down0, conv_w, w_target, eta, chunk,
                   rows, doc_starts=(0,), w_init=None, z=None, target_mode=TARGET_NEXT,
                   clip_tau=None):
    """The same recursion restricted to a subset of W's rows.

    Row i of W, and column i of O, depend on all of Z but only on column i of
    V (W[i] += eta * sum_t V[t,i] Z[t]; O[t,i] = Z[t] . W[i]).  So the sampled
    rows are exact without computing the others.  ``z`` may pass in
    swiglu_intermediate(x, w_gate, w_up) when several runs share the tokens (Z
    does not depend on the chunking or on W).  With ``clip_tau`` the clip scale
    of each chunk needs the whole delta's norm, which is computed in full.
    Returns (O[:, rows], W[rows])."""
    rows = np.asarray(rows, dtype=np.int64)
    x = _f64(x)
    x0 = _f64(x0)
    w0r = _f64(w_down0)[rows]
    wt = _f64(w_target)[:, rows]
    n = x.shape[0]
    W = w0r.copy() if w_init is None else _f64(w_init)[rows].copy()
    out = np.zeros((n, rows.size), dtype=np.float64)
    for s, e, reset in chunk_spans(n, chunk, doc_starts):
        if reset:
            W = w0r.copy()
        zc = swiglu_intermediate(x[s:e], w_gate, w_up) if z is None else _f64(z[s:e])
        out[s:e] = zc @ W.T
        src = chunk_target_source(x0[s:e], conv_w, target_mode)
        v = src @ wt
        scale = 1.0
        if clip_tau:
            nrm = float(np.linalg.norm(float(eta) * ((src @ _f64(w_target)).T @ zc)))
            scale = clip_tau / nrm if nrm > clip_tau else 1.0
        W = W + scale * (float(eta) * (v.T @ zc))
    return out, W


def chunk_delta_norms(x, x0, w_gate, w_up, conv_w, w_target, eta, chunk, doc_starts=(0,),
                      target_mode=TARGET_NEXT, z=None):
    """||eta V_c^T Z_c||_F of every chunk's unclipped delta, in chunk order
    (the quantity the clipping of reading R5 compares with its threshold)."""
    x = _f64(x)
    x0 = _f64(x0)
    out = []
    for s, e, _ in chunk_spans(x.shape[0], chunk, doc_starts):
        zc = swiglu_intermediate(x[s:e], w_gate, w_up) if z is None else _f64(z[s:e])
        v = chunk_target(x0[s:e], conv_w, w_target, target_mode)
        out.append(float(np.linalg.norm(float(eta) * (v.T @ zc))))
    return np.array(out)


def rms_norm(h, eps=1e-6) -> np.ndarray:
    """RMSNorm with unit gain: h / sqrt(mean(h^2) + eps), per row."""
    h = _f64(h)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)


def static_mlp(x, w_gate, w_up, w_down) -> np.ndarray:
    """The ordinary SwiGLU MLP block, Z W_down^T with Z = SiLU(X W_gate^T) *
    (X W_up^T): a block that does not carry TTT ([SUM] C.3; reading R13)."""
    return swiglu_intermediate(x, w_gate, w_up) @ _f64(w_down).T


def ttt_stack(h0, layers, eta, chunk, doc_starts=(0,), eps=1e-6, n_layers=None,
              x0=None, target_mode=TARGET_NEXT, clip_tau=None, ttt_every=1,
              return_states=False):
    """Stack of pre-norm residual SwiGLU MLP blocks (no attention).

    h_{l+1} = h_l + MLP_l(RMSNorm(h_l)) with X0 = h_0 for every TTT block (X0
    is the embedding sequence fed to the stack, [BLOG] 4).  MLP_l is a
    TTT-MLP block when (l + 1) % ttt_every == 0 and the static SwiGLU MLP
    otherwise (reading R13; [SUM] C.3 puts TTT in every sixth block).
    ``x0`` is that embedding sequence as stored for the layers (default: h0
    itself).  Each layer's recursion runs over all tokens before the next
    layer starts; that is the same computation because nothing mixes tokens
    across layers except the per-layer chunk recursion.  Returns (h_L, list of
    the final W per layer; a static block's is its W_down), and with
    ``return_states`` also the list h_0, h_1, ..., h_L."""
    h = _f64(h0).copy()
    x0 = _f64(h0 if x0 is None else x0)
    finals = []
    states = [h.copy()]
    for li, w in enumerate(layers[: n_layers or len(layers)]):
        xn = rms_norm(h, eps)
        if (li + 1) % ttt_every == 0:
            o, wf = ttt_layer(xn, x0, w["w_gate"], w["w_up"], w["w_down0"],
                              w["conv_w"], w["w_target"], eta, chunk, doc_starts,
                              target_mode=target_mode, clip_tau=clip_tau)
        else:
            o, wf = static_mlp(xn, w["w_gate"], w["w_up"], w["w_down0"]), _f64(w["w_down0"])
        h = h + o
        finals.append(wf)
        if return_states:
            states.append(h.copy())
    return (h, finals, states) if return_states else (h, finals)
