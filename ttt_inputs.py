"""Seeded synthetic inputs for the In-Place TTT chunk-wise W_down path.

This module is the one piece of code that both the CPU oracle and the CUDA
path's tests/benchmark use.  It only draws random numbers and rounds them to
the storage precision the GPU sees; it holds none of the method's arithmetic
(no SwiGLU, no convolution, no apply or update).

Recipe (numpy ``default_rng(seed)``, PCG64; float64 standard normals, scaled,
then cast).  Draw order per layer: X, W_gate, W_up, W_down, conv, W_target.

* ``tiny``   d=64, f=256, T=1024, one document, C=64, k=4, eta=0.01, fp32;
             every tensor ~ N(0, 1/fan_in), fan_in = the length the tensor is
             contracted over (X, W_gate, W_up, W_target: d; W_down: f; conv: k).
* ``qwen``   d=2560, f=9728, T=32768, C=256, k=5, eta=1e-3, bf16 storage;
             X ~ N(0,1) with every row RMS-normalised (eps 1e-6, fp32) before
             the bf16 cast; X0 = X; all weights ~ N(0, 0.02^2).
* ``long``   as ``qwen`` with T=131072 and documents starting every 32768.
* ``sweep``  as ``qwen`` with T=16384 per document and per-document X drawn
             from seed 1000+b; shared weights from seed 0.
* ``stack``  L layers of ``qwen``-shaped weights (seed 0, layer-ordered draws),
             h0 ~ N(0,1) (drawn after all layers), T=65536.  At the full 36-layer
             size the weights (2.9 G values) are drawn on the GPU instead
             (``make_stack_device``: torch's device generator seeded with
             seed*1000 + layer, draw order W_gate, W_up, W_down, conv,
             W_target, then h0 from seed*1000 + L); those inputs never meet the
             oracle, only properties that hold at any size.

The same generators take smaller shapes for parity tests (``make_layer``).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "round_bf16",
    "bf16_bits",
    "make_layer_weights",
    "make_tokens",
    "make_layer",
    "make_stack",
    "make_stack_device",
    "CONFIGS",
]


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even); returns float32 values."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) & np.uint32(0xFFFF0000)).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already bf16-exact."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    if np.any(u & np.uint32(0xFFFF)):
        raise ValueError("values are not bf16-representable; call round_bf16 first")
    return (u >> np.uint32(16)).astype(np.uint16)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return (rng.standard_normal(shape) * std).astype(np.float32)


def _store(a: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(a) if dtype == "bf16" else np.ascontiguousarray(a, np.float32)


def make_layer_weights(rng, d: int, f: int, k: int, init: str, dtype: str) -> dict:
    """W_gate, W_up (f x d), W_down (d x f), conv (k x d), W_target (d x d).

    ``init`` is "fan_in" (variance 1/fan_in) or a float standard deviation.
    Layouts follow nn.Linear (out x in); W_target is in x out (V = U W_target).
    """
    def std(fan_in):
        return (1.0 / fan_in) ** 0.5 if init == "fan_in" else float(init)

    w = {}
    w["w_gate"] = _store(_normal(rng, (f, d), std(d)), dtype)
    w["w_up"] = _store(_normal(rng, (f, d), std(d)), dtype)
    w["w_down0"] = _store(_normal(rng, (d, f), std(f)), dtype)
    w["conv_w"] = _store(_normal(rng, (k, d), std(k)), dtype)
    w["w_target"] = _store(_normal(rng, (d, d), std(d)), dtype)
    return w


def make_tokens(rng, T: int, d: int, mode: str, dtype: str) -> np.ndarray:
    """Token inputs X (T x d): ``mode`` "fan_in" (N(0,1/d)), "rms" (N(0,1) rows
    RMS-normalised in fp32 with eps 1e-6) or "normal" (N(0,1))."""
    if mode == "fan_in":
        x = _normal(rng, (T, d), (1.0 / d) ** 0.5)
    else:
        x = rng.standard_normal((T, d)).astype(np.float32)
        if mode == "rms":
            ms = np.mean(x.astype(np.float32) ** 2, axis=1, keepdims=True, dtype=np.float32)
            x = (x / np.sqrt(ms + np.float32(1e-6))).astype(np.float32)
    return _store(x, dtype)


def make_layer(d: int, f: int, T: int, chunk: int, k: int, eta: float,
               dtype: str = "bf16", seed: int = 0, init="qwen",
               doc_starts=(0,), x_seed=None) -> dict:
    """One TTT-MLP layer workload.

    init="tiny": every tensor N(0,1/fan_in) (X drawn first, then the weights).
    init="qwen": X ~ N(0,1) rows RMS-normalised, weights N(0, 0.02^2).
    ``x_seed`` (if given) draws X from its own generator (per-document inputs
    of the batch sweep) after the weights come from ``seed``.
    """
    rng = np.random.default_rng(seed)
    if init == "tiny":
        x_mode, w_init = "fan_in", "fan_in"
    else:
        x_mode, w_init = "rms", 0.02
    if x_seed is None:
        x = make_tokens(rng, T, d, x_mode, dtype)
        w = make_layer_weights(rng, d, f, k, w_init, dtype)
    else:
        w = make_layer_weights(rng, d, f, k, w_init, dtype)
        x = make_tokens(np.random.default_rng(x_seed), T, d, x_mode, dtype)
    cfg = dict(d=d, f=f, T=T, chunk=chunk, k=k, eta=float(eta), dtype=dtype,
               doc_starts=tuple(int(s) for s in doc_starts))
    cfg.update(w)
    cfg["x"] = x
    cfg["x0"] = x
    return cfg


def make_stack(n_layers: int, d: int, f: int, T: int, chunk: int, k: int, eta: float,
               seed: int = 0, dtype: str = "bf16"):
    """Stack workload: returns (h0 float32 T x d, list of per-layer weight dicts).
    Layer weights are drawn in layer order from one generator, then h0 ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    layers = [make_layer_weights(rng, d, f, k, 0.02, dtype) for _ in range(n_layers)]
    h0 = rng.standard_normal((T, d)).astype(np.float32)
    meta = dict(d=d, f=f, T=T, chunk=chunk, k=k, eta=float(eta), dtype=dtype)
    return h0, layers, meta


def make_stack_device(n_layers: int, d: int, f: int, T: int, k: int, seed: int = 0,
                      device="cuda", dtype=None):
    """Full-size stack inputs drawn on the GPU: (h0 fp32 T x d, list of
    per-layer weight dicts of `dtype` (default bf16) CUDA tensors)."""
    import torch
    dt = dtype or torch.bfloat16
    layers = []
    for li in range(n_layers):
        g = torch.Generator(device=device).manual_seed(seed * 1000 + li)

        def nrm(*shape):
            return (torch.randn(*shape, generator=g, device=device) * 0.02).to(dt)

        layers.append({"w_gate": nrm(f, d), "w_up": nrm(f, d), "w_down0": nrm(d, f),
                       "conv_w": nrm(k, d), "w_target": nrm(d, d)})
    g = torch.Generator(device=device).manual_seed(seed * 1000 + n_layers)
    h0 = torch.randn(T, d, generator=g, device=device)
    return h0, layers


# Named workloads (sizes of the five measured configurations).
CONFIGS = {
    "tiny": dict(d=64, f=256, T=1024, chunk=64, k=4, eta=0.01, dtype="f32", init="tiny"),
    "qwen": dict(d=2560, f=9728, T=32768, chunk=256, k=5, eta=1e-3, dtype="bf16", init="qwen"),
    "long": dict(d=2560, f=9728, T=131072, chunk=256, k=5, eta=1e-3, dtype="bf16", init="qwen",
                 doc_starts=(0, 32768, 65536, 98304)),
    "sweep": dict(d=2560, f=9728, T=16384, chunk=256, k=5, eta=1e-3, dtype="bf16", init="qwen"),
    "stack": dict(n_layers=36, d=2560, f=9728, T=65536, chunk=256, k=5, eta=1e-3, dtype="bf16"),
}
