"""Seeded synthetic inputs shaped like the C2KV RAG workloads.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic (no positions, no rotation, no attention).  Both the
CUDA path and the CPU oracle are fed from the same arrays it returns, so the
two sides see identical bf16 bytes.

Workload shapes follow the multi-document QA setting of the C2KV explainer
(paper-daily.com, section "pipeline: extract, store, concatenate") and the
attention geometries of the base models it names (Llama3.1-8B, Qwen3-14B,
section "limitations").  No dataset is used: every value is drawn from a
seeded PCG64 stream.

Value recipe: K/V/q ~ N(0, 1) in fp32, rounded to bf16 (round to nearest
even).  Each document's stream is keyed by (seed, doc_id) so a document
drawn into several requests carries the same bytes every time.  All bf16
arrays are returned as ``numpy.uint16`` bit patterns.

Segment layout (host and device): ``[layer][kv_head][slot][head_dim]``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Geometry:
    """Attention geometry of one base model."""
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    rope_theta: float

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


LLAMA31_8B = Geometry(32, 32, 8, 128, 5.0e5)
QWEN3_14B = Geometry(40, 40, 8, 128, 1.0e6)
TINY = Geometry(1, 4, 2, 64, 1.0e4)


@dataclass(frozen=True)
class Workload:
    """One request mix: documents, compression ratio, question and decode."""
    name: str
    geom: Geometry
    k: int                      # document tokens per compressed slot
    batch: int                  # requests decoded together
    q_len: int                  # question tokens prefilled per request
    decode_steps: int           # answer tokens decoded per request
    doc_tokens: tuple = ()      # fixed per-request document lengths (if no pool)
    pool_docs: int = 0          # >0: requests draw from a shared pool
    pool_len_range: tuple = ()  # (lo, hi) uniform, multiples of k
    docs_per_request: int = 0
    seed: int = 0xC2C0


WORKLOADS: Dict[str, Workload] = {
    # 3 documents of 12/400/40 tokens at k=4 -> 3/100/10 slots.
    "tiny": Workload("tiny", TINY, k=4, batch=1, q_len=8, decode_steps=16,
                     doc_tokens=(12, 400, 40), seed=0xC2C0),
    # 8 documents x 4000 tokens at k=4 -> 8000 composed slots.
    "llama8b_8x4000_k4": Workload("llama8b_8x4000_k4", LLAMA31_8B, k=4,
                                  batch=1, q_len=64, decode_steps=128,
                                  doc_tokens=(4000,) * 8, seed=0xC2C1),
    # 16 requests, each 8 documents drawn from a 256-document pool.
    "llama8b_pool256_b16_k4": Workload("llama8b_pool256_b16_k4", LLAMA31_8B,
                                       k=4, batch=16, q_len=32,
                                       decode_steps=64, pool_docs=256,
                                       pool_len_range=(500, 4000),
                                       docs_per_request=8, seed=0xC2C2),
    # 32 documents x 4096 tokens (131072 original tokens) -> 32768 slots.
    "llama8b_32x4096_k4_b4": Workload("llama8b_32x4096_k4_b4", LLAMA31_8B,
                                      k=4, batch=4, q_len=0,
                                      decode_steps=256,
                                      doc_tokens=(4096,) * 32, seed=0xC2C3),
    # Qwen3-14B geometry, 16 documents x 8000 tokens at k=16 -> 8000 slots.
    "qwen14b_16x8000_k16_b8": Workload("qwen14b_16x8000_k16_b8", QWEN3_14B,
                                       k=16, batch=8, q_len=128,
                                       decode_steps=128,
                                       doc_tokens=(8000,) * 16, seed=0xC2C4),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(scale))


def synthetic_slots(n_tokens: int, k: int) -> int:
    """Slots an extractor with one slot per k-token block emits for a document.

    This fixes the *shape* of the synthetic segments only; the library never
    derives slot counts itself (the caller records them in the store).
    """
    return -(-n_tokens // k)


@dataclass
class Document:
    doc_id: int
    n_tokens: int
    n_slots: int
    k_pre: np.ndarray   # uint16 [L][Hkv][n_slots][d], pre-RoPE
    v: np.ndarray       # uint16 [L][Hkv][n_slots][d]


def make_document(geom: Geometry, doc_id: int, n_tokens: int, k: int,
                  seed: int, n_slots: Optional[int] = None,
                  layers: Optional[int] = None) -> Document:
    """Draw one document's compressed pre-RoPE segment."""
    s = synthetic_slots(n_tokens, k) if n_slots is None else n_slots
    L = geom.n_layers if layers is None else layers
    rng = _rng(seed, 0xD0C, doc_id)
    shape = (L, geom.n_kv_heads, s, geom.head_dim)
    return Document(doc_id, n_tokens, s, normal_bf16(rng, shape),
                    normal_bf16(rng, shape))


@dataclass
class Request:
    doc_ids: List[int]          # documents in request (retrieval) order
    order: Optional[List[int]]  # permutation into doc_ids; None = identity


def make_requests(w: Workload) -> tuple:
    """Return (docs: {doc_id: (n_tokens, n_slots)}, [Request] * batch)."""
    rng = _rng(w.seed, 0x9E0)
    docs: Dict[int, tuple] = {}
    reqs: List[Request] = []
    if w.pool_docs:
        lo, hi = w.pool_len_range
        choices = np.arange(lo, hi + 1, w.k)
        lens = rng.choice(choices, size=w.pool_docs)
        for i in range(w.pool_docs):
            docs[i] = (int(lens[i]), synthetic_slots(int(lens[i]), w.k))
        for _ in range(w.batch):
            ids = rng.choice(w.pool_docs, size=w.docs_per_request, replace=False)
            perm = rng.permutation(w.docs_per_request)
            reqs.append(Request([int(i) for i in ids], [int(p) for p in perm]))
    else:
        ids = list(range(len(w.doc_tokens)))
        for i, n in zip(ids, w.doc_tokens):
            docs[i] = (int(n), synthetic_slots(int(n), w.k))
        for b in range(w.batch):
            perm = None if b == 0 else [int(p) for p in rng.permutation(len(ids))]
            reqs.append(Request(list(ids), perm))
    return docs, reqs


@dataclass
class StepInputs:
    """Per-layer question and decode inputs for one batch of requests."""
    q_pre: np.ndarray      # uint16 [L][B][Q][Hq][d]
    kq_pre: np.ndarray     # uint16 [L][B][Q][Hkv][d]
    vq: np.ndarray         # uint16 [L][B][Q][Hkv][d]
    qd_pre: np.ndarray     # uint16 [T][L][B][Hq][d]
    kd_pre: np.ndarray     # uint16 [T][L][B][Hkv][d]
    vd: np.ndarray         # uint16 [T][L][B][Hkv][d]


def make_step_inputs(w: Workload, layers: Optional[int] = None,
                     decode_steps: Optional[int] = None,
                     q_scale: float = 1.0) -> StepInputs:
    g = w.geom
    L = g.n_layers if layers is None else layers
    T = w.decode_steps if decode_steps is None else decode_steps
    rng = _rng(w.seed, 0x057E)
    B, Q, d = w.batch, w.q_len, g.head_dim
    return StepInputs(
        normal_bf16(rng, (L, B, Q, g.n_q_heads, d), q_scale),
        normal_bf16(rng, (L, B, Q, g.n_kv_heads, d)),
        normal_bf16(rng, (L, B, Q, g.n_kv_heads, d)),
        normal_bf16(rng, (T, L, B, g.n_q_heads, d), q_scale),
        normal_bf16(rng, (T, L, B, g.n_kv_heads, d)),
        normal_bf16(rng, (T, L, B, g.n_kv_heads, d)),
    )


# ---------------------------------------------------------------- decoder step
@dataclass(frozen=True)
class ModelShape:
    """Sizes of a decoder stack around the attention geometry: hidden size,
    MLP width, vocabulary, RMSNorm epsilon (Llama-3.1-8B's published sizes)."""
    dim: int
    ffn: int
    vocab: int
    eps: float


LLAMA31_8B_MODEL = ModelShape(4096, 14336, 128256, 1e-5)


def make_decoder_weights(geom: Geometry, shape: ModelShape, layers: int, seed: int,
                         lm_head: bool = False) -> dict:
    """Seeded bf16 weights (uint16 bit patterns) of `layers` decoder layers:
    norms 1 + 0.1 N(0,1), projections N(0, 1/fan_in) so activations stay O(1).
    Per layer: attn_norm [dim], qkv [(Hq + 2 Hkv) d][dim], o [dim][Hq d],
    mlp_norm [dim], gate_up [2 ffn][dim] (gate and up rows in 64-row blocks),
    down [dim][ffn]; with lm_head also final_norm [dim] and lm_head
    [vocab][dim]."""
    d, dim, F = geom.head_dim, shape.dim, shape.ffn
    nq, nkv = geom.n_q_heads * d, geom.n_kv_heads * d
    out = {"layers": []}
    for l in range(layers):
        rng = _rng(seed, 0xDEC, l)
        out["layers"].append({
            "attn_norm": bf16_bits(1.0 + 0.1 * rng.standard_normal(dim, dtype=np.float32)),
            "qkv": normal_bf16(rng, (nq + 2 * nkv, dim), dim ** -0.5),
            "o": normal_bf16(rng, (dim, nq), nq ** -0.5),
            "mlp_norm": bf16_bits(1.0 + 0.1 * rng.standard_normal(dim, dtype=np.float32)),
            "gate_up": normal_bf16(rng, (2 * F, dim), dim ** -0.5),
            "down": normal_bf16(rng, (dim, F), F ** -0.5),
        })
    if lm_head:
        rng = _rng(seed, 0xDEC, 0xFFFF)
        out["final_norm"] = bf16_bits(1.0 + 0.1 * rng.standard_normal(dim, dtype=np.float32))
        out["lm_head"] = normal_bf16(rng, (shape.vocab, dim), dim ** -0.5)
    return out
