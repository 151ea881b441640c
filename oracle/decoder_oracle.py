"""Plain CPU oracle of the synthetic-weight decoder step around the attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only the tests, the package smoke check and the benchmark's CPU
baseline leg use it.  It shares no code with the CUDA library.

C2KV explainer (paper-daily.com), section "the problem" (它到底在解决什么问题？),
Fig. 1: the time to first token and the decode rate of the whole model are
what the cache reuse buys; the base models it names (Llama3.1-8B, Qwen3-14B,
section "limitations") are standard pre-norm decoder stacks.  The pages do
not describe the layer, so this follows the plainest reading (D17): a
Llama-3 decoder layer without biases,
    h = rmsnorm(x) * w_attn;  q, k, v = h W_q^T, h W_k^T, h W_v^T
    x = x + attention(q, k, v over the composed cache) W_o^T
    h = rmsnorm(x) * w_mlp;   x = x + (silu(h W_g^T) * (h W_u^T)) W_d^T
with rmsnorm(x) = x / sqrt(mean(x^2) + eps), silu(g) = g / (1 + e^-g).

Everything is fp64 numpy.  Activations are rounded to bf16 at the points
where a bf16 model stores them (after each norm, each projection, the
attention output and each residual update), with the oracle's own
rounding (c2kv_oracle.f64_to_bf16).  Fused gate/up weights use the library's
layout: rows 128i .. 128i+63 are the gate rows of features 64i .. 64i+63,
rows 128i+64 .. 128i+127 their up rows.

Parity pins: tests/test_oracle_pins.py (closed forms, brute force at tiny
sizes, the zero-weight identity of a layer).
"""
from __future__ import annotations

import numpy as np

from . import c2kv_oracle as O  # noqa: N812 (also reached as decoder_oracle.O)


def rms_norm(x_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """x bits [t][dim], w bits [dim] -> fp64 [t][dim]."""
    x = O.bf16_to_f64(x_bits)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / r * O.bf16_to_f64(w_bits)[None, :]


def linear(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """x bits [t][k], w bits [n][k] -> fp64 x W^T [t][n]."""
    return O.bf16_to_f64(x_bits) @ O.bf16_to_f64(w_bits).T


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def split_gate_up(w_gu_bits: np.ndarray):
    """The fused [2F][k] gate/up weight -> (gate [F][k], up [F][k]) bits."""
    n2, k = w_gu_bits.shape
    blocks = w_gu_bits.reshape(n2 // 128, 2, 64, k)
    return blocks[:, 0].reshape(-1, k), blocks[:, 1].reshape(-1, k)


def swiglu(h_bits: np.ndarray, w_gu_bits: np.ndarray) -> np.ndarray:
    """silu(h W_g^T) * (h W_u^T), fp64 [t][F]."""
    wg, wu = split_gate_up(w_gu_bits)
    return silu(linear(h_bits, wg)) * linear(h_bits, wu)


def bf16(x: np.ndarray) -> np.ndarray:
    return O.f64_to_bf16(x)


def decoder_layer_decode(x_bits, w, k_caches, v_caches, start_pos, theta, n_q_heads, n_kv_heads, eps):
    """One decode step of one layer for a batch of sequences, one token each.

    x_bits [B][dim] (bf16 residual stream), w: dict of bf16 weights
    ("attn_norm" [dim], "qkv" [(Hq + 2 Hkv) d][dim], "o" [dim][Hq d],
    "mlp_norm" [dim], "gate_up" [2F][dim], "down" [dim][F]); k_caches[b],
    v_caches[b]: bits [Hkv][n_b][d] of sequence b's composed cache (keys
    rotated); start_pos[b]: the new token's position.  Returns the new
    residual stream bits [B][dim] and the per-stage bf16 activations (for
    stage-wise checks)."""
    B, dim = x_bits.shape
    d = dim // n_q_heads
    nq, nkv = n_q_heads * d, n_kv_heads * d
    h = bf16(rms_norm(x_bits, w["attn_norm"], eps))
    qkv = bf16(linear(h, w["qkv"]))
    q, k, v = qkv[:, :nq], qkv[:, nq:nq + nkv], qkv[:, nq + nkv:]
    att = np.empty((B, nq), dtype=np.uint16)
    for b in range(B):
        out, _ = O.attend_new_tokens(q[b].reshape(1, n_q_heads, d), k[b].reshape(1, n_kv_heads, d),
                                     v[b].reshape(1, n_kv_heads, d), k_caches[b], v_caches[b],
                                     start_pos[b], theta)
        att[b] = bf16(out[0].reshape(nq))
    x1 = bf16(O.bf16_to_f64(x_bits) + linear(att, w["o"]))
    h2 = bf16(rms_norm(x1, w["mlp_norm"], eps))
    m = bf16(swiglu(h2, w["gate_up"]))
    x2 = bf16(O.bf16_to_f64(x1) + linear(m, w["down"]))
    return x2, {"h": h, "q": q, "k": k, "v": v, "att": att, "x1": x1, "h2": h2, "m": m}
