"""fp64 oracle of a small pre-norm GQA decoder (the Qwen3-8B layer structure).

TEST INFRASTRUCTURE.  Only tests/ (and the smoke check / CPU baseline of the
benchmark) may use it; it shares no code with the CUDA library.

Plain definitions, evaluated in float64 on the host, with the result of every
operation rounded once to bf16 where the GPU path stores bf16:

  embedding        x = E[token]
  per layer l      n   = bf16(rmsnorm(r, w_in))                 (r: residual stream)
                   qkv = bf16(n W_qkv^T)
                   q_h = bf16(rope(bf16(rmsnorm_128(q_h, w_qn)), pos))   per query head
                   k_h = bf16(rope(bf16(rmsnorm_128(k_h, w_kn)), pos))   per kv head
                   a   = bf16(causal softmax(q k^T / sqrt(128)) v)        (GQA: head i uses kv head i // 4)
                   o   = bf16(a W_o^T)
                   r   = bf16(r + o);   n2 = bf16(rmsnorm(r, w_post))
                   gu  = bf16(n2 W_gu^T);  h = bf16(silu(g) * u)   (g, u = halves of gu)
                   d   = bf16(h W_down^T);  r = bf16(r + d)
  final            logits = bf16(rmsnorm(r, w_final)) W_lm^T      (left in fp64)

rope (rotate-half): for i < 64, angle = pos * theta^(-i/64),
    y_i = x_i cos - x_{64+i} sin,   y_{64+i} = x_{64+i} cos + x_i sin.
silu(g) = g / (1 + exp(-g)).

Sources: the three reduction ops follow "Defeating Nondeterminism in LLM
Inference: The Core Role of Batch Invariance" (sections 1-3); the layer
structure is the Qwen3-8B shape the workload names (pre-norm, GQA 32/8,
head_dim 128, SwiGLU, RoPE theta 1e6, per-head q/k RMSNorm).
Pins: tests/test_oracle.py (rope, silu, causal attention closed forms; for the
composition: a layer whose output projections are zero is the identity, the
zero-layer closed form for a constant embedding row, causality).
"""
from __future__ import annotations

import math

import numpy as np

from . import bf16_to_f64, gemm, rmsnorm, round_bf16


def _b(x64: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 and return them as fp64 again."""
    return bf16_to_f64(round_bf16(x64))


def _bits_of(x64_bf16_exact: np.ndarray) -> np.ndarray:
    """fp64 values that are exactly bf16 -> their uint16 patterns."""
    return round_bf16(x64_bf16_exact)


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of x [..., T, 128] at positions pos [T], fp64."""
    D = x.shape[-1]
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * np.power(float(theta), -i / half)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g)) * u


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """q [T, Hq, D], k, v [T, Hkv, D]; row t attends to keys 0..t of the same
    sequence; query head i uses kv head i // (Hq / Hkv).  fp64."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    out = np.zeros_like(q)
    for i in range(Hq):
        g = i // grp
        s = (q[:, i, :] @ k[:, g, :].T) * scale  # [T, T]
        s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, i, :] = p @ v[:, g, :]
    return out


def _rmsnorm_rows(x64: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """rmsnorm of bf16-exact fp64 rows (any leading shape), rounded to bf16."""
    shp = x64.shape
    rows = x64.reshape(-1, shp[-1])
    return _b(rmsnorm(_bits_of(rows), w_bits, eps)).reshape(shp)


def _linear(x64: np.ndarray, W_bits: np.ndarray) -> np.ndarray:
    return _b(gemm(_bits_of(x64), W_bits))


def forward_logits(weights: dict, tokens: np.ndarray, n_layers: int, Hq: int = 32, Hkv: int = 8,
                   theta: float = 1e6, eps: float = 1e-6, positions=None) -> np.ndarray:
    """Logits [len(positions), vocab] (fp64; all T positions by default) of one
    sequence `tokens` [T] through the first n_layers layers; every position
    sees itself and the ones before.

    `weights`: uint16 bf16 bit patterns: embed [V, H], final_norm [H], lm_head [V, H], and per
    layer l: f"{l}.in_norm" [H], f"{l}.qkv" [(Hq+2Hkv)*128, H], f"{l}.q_norm" [128],
    f"{l}.k_norm" [128], f"{l}.o" [H, Hq*128], f"{l}.post_norm" [H], f"{l}.gate_up" [2F, H],
    f"{l}.down" [H, F]."""
    D = 128
    T = len(tokens)
    pos = np.arange(T)
    r = bf16_to_f64(weights["embed"][np.asarray(tokens)])
    for l in range(n_layers):
        n = _rmsnorm_rows(r, weights[f"{l}.in_norm"], eps)
        qkv = _linear(n, weights[f"{l}.qkv"])
        q = qkv[:, :Hq * D].reshape(T, Hq, D)
        k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D)
        v = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)
        q = _rmsnorm_rows(q, weights[f"{l}.q_norm"], eps)
        k = _rmsnorm_rows(k, weights[f"{l}.k_norm"], eps)
        q = _b(rope(q.transpose(1, 0, 2), pos, theta).transpose(1, 0, 2))
        k = _b(rope(k.transpose(1, 0, 2), pos, theta).transpose(1, 0, 2))
        a = _b(causal_attention(q, k, v, 1.0 / math.sqrt(D)))
        o = _linear(a.reshape(T, Hq * D), weights[f"{l}.o"])
        r = _b(r + o)
        n2 = _rmsnorm_rows(r, weights[f"{l}.post_norm"], eps)
        gu = _linear(n2, weights[f"{l}.gate_up"])
        F = gu.shape[1] // 2
        h = _b(silu_mul(gu[:, :F], gu[:, F:]))
        d = _linear(h, weights[f"{l}.down"])
        r = _b(r + d)
    nf = _rmsnorm_rows(r, weights["final_norm"], eps)
    if positions is not None:
        nf = nf[np.asarray(positions)]
    return gemm(_bits_of(nf), weights["lm_head"])
