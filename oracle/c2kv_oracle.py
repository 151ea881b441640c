"""Plain CPU oracle for the C2KV composed-cache hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only the tests, the package smoke check and the benchmark's CPU
baseline leg use it.  It shares no code with the CUDA library.

Everything is fp64 numpy, written step by step from the definitions on the
pages (no blocking, fusion or reordering):

* C2KV explainer, "C 2 KV: Compressed and Composable KV Cache Reuse for
  Efficient LLM Inference" (paper-daily.com):
    - section "positions at concatenation" (拼接时位置怎么处理？): stored
      K/V are pre-RoPE; at extraction slot j sits at the last token of its
      k-token block; at composition every segment keeps its original length
      of positions and each document is shifted by the summed original
      lengths of the documents before it.
    - section "pipeline: extract, store, concatenate" (整体流程): fetch,
      re-apply position encoding, concatenate, append the question and
      generate; no repair step.
    - section "structured information flow" (为什么需要“结构化信息流”？) and
      its k=4 figure: the three mask rules.
* arXiv 2607.17715 listing (arxivdaily.com), English abstract: the cache is
  composed without modifying the frozen base model.

Readings where the pages are silent (each listed in the design notes):
  S1  a document of n tokens at ratio k carries ceil(n/k) slots; the last
      slot of a partial block sits at the document's last token.
  S2  RoPE is the rotate-half form with inv_freq_i = theta^(-2i/d), fp64.
  S3  question token i sits at L_tot + i (original composed length).
  S4  ``order`` is a permutation into doc_ids; None means identity.
  S9  softmax scale is 1/sqrt(d).
  S11 re-rotated K is stored as bf16, rounded to nearest even.
  S15 the "no position re-alignment" ablation (section "results") keeps
      every document at its extraction positions (no offset off_c); the
      question still starts at L_tot.
  S16 the "anchor tokens" ablation (section "results") swaps only the mask
      of the extraction pass: the extra tokens sit where the slots sit and
      see every document token, and every document token sees every extra
      token as well as its causal prefix of the document; the extra tokens
      see each other causally, as the slots do.

Parity pins: every function below is checked by tests/test_oracle_pins.py
against the pages' worked values, closed forms, invariants or brute force.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# ---------------------------------------------------------------------------
# bf16 <-> fp64 (the oracle's own conversions)
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (nearest, ties to even); returns uint16 bits.

    bf16 keeps 8 significant bits and fp32's exponent range.  A finite value
    with |x| in [2^(e-1), 2^e) is rounded to a multiple of 2^(e-8); below the
    normal range (e-1 < -126) the quantum stays 2^-133.  Scaling by powers of
    two is exact, so the only rounding is np.rint, which breaks ties to even.
    Rounding directly from fp64 avoids double rounding through fp32.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    finite = np.isfinite(x)
    xf = x[finite]
    _, e = np.frexp(xf)
    quantum_exp = np.maximum(e, -125) - 8
    q = np.ldexp(np.rint(np.ldexp(xf, -quantum_exp)), quantum_exp)
    # q is exactly representable in bf16 (or overflows to +-inf in fp32).
    with np.errstate(over="ignore"):
        q32 = q.astype(np.float32)
    out[finite] = (q32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nonfinite = ~finite
    if nonfinite.any():
        bad = x[nonfinite]
        nb = np.where(np.isnan(bad), 0x7FC0, np.where(bad > 0, 0x7F80, 0xFF80))
        out[nonfinite] = nb.astype(np.uint16)
    return out


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units of last place between two bf16 bit arrays."""
    def ordered(bits):
        v = np.asarray(bits, dtype=np.uint16).astype(np.int32)
        return np.where(v & 0x8000, 0x8000 - v, v)   # monotone in the real value
    return np.abs(ordered(a_bits) - ordered(b_bits))


# ---------------------------------------------------------------------------
# Positions (C2KV explainer, section "positions at concatenation")
# ---------------------------------------------------------------------------


def slot_count(n_tokens: int, k: int) -> int:
    """One slot per k-token block (section "C2 tokens"); reading S1 for a
    partial last block."""
    return -(-n_tokens // k)


def extraction_slot_position(j: int, n_tokens: int, k: int) -> int:
    """Position id of slot j (0-based) at extraction: the last token of the
    block it summarises, i.e. (j+1)k-1, clipped to the document's last token
    for a partial block (reading S1)."""
    return min((j + 1) * k, n_tokens) - 1


def composed_positions(n_tokens: Sequence[int], n_slots: Sequence[int],
                       k: int, realign: bool = True) -> Tuple[np.ndarray, int]:
    """Position of every composed slot, documents taken in composed order.

    Each document occupies its original length of positions; document d's
    slots are shifted by off_d = sum of the original lengths before it.
    realign=False is the ablation without that shift (reading S15): every
    document keeps its extraction positions.
    Returns (int64 positions [sum n_slots], L_tot = sum n_tokens)."""
    pos: List[int] = []
    off = 0
    for n, s in zip(n_tokens, n_slots):
        for j in range(s):
            pos.append((off if realign else 0) + extraction_slot_position(j, n, k))
        off += n
    return np.asarray(pos, dtype=np.int64), off


def composed_order(doc_ids: Sequence[int], order: Optional[Sequence[int]]) -> List[int]:
    """Documents in composed order (reading S4: order[i] indexes doc_ids)."""
    if order is None:
        return list(doc_ids)
    return [doc_ids[o] for o in order]


# ---------------------------------------------------------------------------
# RoPE (reading S2: rotate-half, fp64)
# ---------------------------------------------------------------------------


def rope_inv_freq(theta: float, d: int) -> np.ndarray:
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / d)


def rope_rotate(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate x[..., n, d] (fp64) by RoPE at positions pos[n].

    Pair (i, i + d/2) is rotated by angle pos * inv_freq_i:
        x'_i       = x_i cos a - x_{i+d/2} sin a
        x'_{i+d/2} = x_{i+d/2} cos a + x_i sin a
    """
    d = x.shape[-1]
    h = d // 2
    a = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(theta, d)[None, :]
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# Composition (sections "pipeline" and "positions at concatenation")
# ---------------------------------------------------------------------------

StoreDoc = Tuple[int, int, np.ndarray, np.ndarray]  # (n_tokens, n_slots, k_pre, v)


def compose(store: Dict[int, StoreDoc], doc_ids: Sequence[int],
            order: Optional[Sequence[int]], k: int, theta: float,
            layers: Optional[Sequence[int]] = None, realign: bool = True):
    """Compose one request's cache from stored pre-RoPE segments.

    store[doc_id] = (n_tokens, n_slots, k_pre bits [L][Hkv][s][d],
    v bits [L][Hkv][s][d]).  Returns (pos int64 [N], L_tot,
    K_rot bits [len(layers)][Hkv][N][d], V bits [len(layers)][Hkv][N][d]).
    The segments are concatenated in composed order; K is rotated at the
    remapped positions and rounded to bf16 (reading S11); V is copied."""
    seq = composed_order(doc_ids, order)
    n_tok = [store[d][0] for d in seq]
    n_sl = [store[d][1] for d in seq]
    pos, l_tot = composed_positions(n_tok, n_sl, k, realign)
    if not store:
        raise ValueError("empty store")
    L, hkv, _, d = next(iter(store.values()))[2].shape   # every stored segment has this geometry
    layers = list(range(L)) if layers is None else list(layers)
    # no documents: the concatenation of no segments, a cache of 0 rows
    k_cat = np.concatenate([np.zeros((len(layers), hkv, 0, d), np.uint16)] +
                           [store[d_][2][layers] for d_ in seq], axis=2)
    v_cat = np.concatenate([np.zeros((len(layers), hkv, 0, d), np.uint16)] +
                           [store[d_][3][layers] for d_ in seq], axis=2)
    k_rot = f64_to_bf16(rope_rotate(bf16_to_f64(k_cat), pos, theta))
    return pos, l_tot, k_rot, v_cat.copy()


# ---------------------------------------------------------------------------
# Attention (plain masked softmax, reading S9)
# ---------------------------------------------------------------------------


def masked_softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                             mask: np.ndarray) -> np.ndarray:
    """q [r][d], K [n][d], V [n][d], mask [r][n] (True = visible), all fp64.

    out_i = sum_j p_ij V_j with p_i = softmax over visible j of q_i.K_j/sqrt(d),
    computed with the row maximum subtracted."""
    d = q.shape[-1]
    s = (q @ K.T) / math.sqrt(d)
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        raise ValueError("a query row sees no key")
    p = np.exp(s - m)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ V


def rotate_keys_bf16(k_pre: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate new keys k_pre bits [t][Hkv][d] at positions pos[t] and round
    them to bf16 as they are stored in the cache: returns bits [Hkv][t][d]."""
    return f64_to_bf16(rope_rotate(bf16_to_f64(k_pre).transpose(1, 0, 2), pos, theta))


def attend_new_tokens(q_pre: np.ndarray, k_new_pre: np.ndarray, v_new: np.ndarray,
                      k_cache: np.ndarray, v_cache: np.ndarray,
                      start_pos: int, theta: float):
    """Append t new tokens after a cache of n keys and attend causally (GQA).

    q_pre bits [t][Hq][d], k_new_pre/v_new bits [t][Hkv][d] (pre-RoPE),
    k_cache/v_cache bits [Hkv][n][d] (k already rotated).  Token i sits at
    position start_pos + i (reading S3 for the question; the decode step
    continues the count) and sees every cached key plus new tokens 0..i.
    q head h reads kv head h // (Hq/Hkv).  The new keys are rotated and
    rounded to bf16 as they are stored in the cache; q is rotated in fp64
    and not rounded.  Returns (out fp64 [t][Hq][d], k_new_rot bits
    [Hkv][t][d]).
    """
    t, hq, d = q_pre.shape
    hkv = k_new_pre.shape[1]
    g = hq // hkv
    n = k_cache.shape[1]
    pos = start_pos + np.arange(t, dtype=np.int64)
    q = rope_rotate(bf16_to_f64(q_pre).transpose(1, 0, 2), pos, theta)   # [Hq][t][d]
    k_new_rot = rotate_keys_bf16(k_new_pre, pos, theta)
    K = np.concatenate([bf16_to_f64(k_cache), bf16_to_f64(k_new_rot)], axis=1)
    V = np.concatenate([bf16_to_f64(v_cache), bf16_to_f64(v_new).transpose(1, 0, 2)], axis=1)
    mask = np.arange(n + t)[None, :] < (n + 1 + np.arange(t))[:, None]
    out = np.empty((t, hq, d), dtype=np.float64)
    for h in range(hq):
        out[:, h, :] = masked_softmax_attention(q[h], K[h // g], V[h // g], mask)
    return out, k_new_rot


def decode_sequence(qd_pre, kd_pre, vd, k_cache, v_cache, start_pos, theta):
    """T decode steps for one layer of one sequence: step t appends its token
    at start_pos + t and attends over everything cached so far plus itself.
    qd_pre bits [T][Hq][d], kd_pre/vd bits [T][Hkv][d].
    Returns (out fp64 [T][Hq][d], final k_cache bits, final v_cache bits)."""
    T = qd_pre.shape[0]
    outs = []
    kc, vc = k_cache, v_cache
    for t in range(T):
        o, krot = attend_new_tokens(qd_pre[t:t + 1], kd_pre[t:t + 1], vd[t:t + 1],
                                    kc, vc, start_pos + t, theta)
        outs.append(o[0])
        kc = np.concatenate([kc, krot], axis=1)
        vc = np.concatenate([vc, vd[t:t + 1].transpose(1, 0, 2)], axis=1)
    return np.stack(outs), kc, vc


# ---------------------------------------------------------------------------
# Structured information flow (extraction-time mask)
# ---------------------------------------------------------------------------


def structured_mask(n_doc: int, n_slot: int, k: int) -> np.ndarray:
    """Mask over n_doc document tokens followed by n_slot slots
    (rows = queries, columns = keys, True = visible).

    Rule 1: document tokens keep the base causal mask and never see slots.
    Rule 2: slot i sees the sink block B(0) -- the document's first k tokens --
            and its own block, tokens [i*k, min((i+1)k, n_doc)).
    Rule 3: slot i sees slots 0..i (causal, including itself).
    The slots are drawn after the document only for the figure; their
    positions come from extraction_positions()."""
    N = n_doc + n_slot
    m = np.zeros((N, N), dtype=bool)
    for r in range(n_doc):
        m[r, :r + 1] = True
    for i in range(n_slot):
        row = n_doc + i
        m[row, :min(k, n_doc)] = True
        m[row, i * k:min((i + 1) * k, n_doc)] = True
        m[row, n_doc:n_doc + i + 1] = True
    return m


def anchor_mask(n_doc: int, n_slot: int) -> np.ndarray:
    """Mask of the "anchor tokens" ablation (reading S16) over n_doc document
    tokens followed by n_slot anchor tokens (True = visible).

    Documents and anchors see each other in both directions: document token r
    sees document tokens 0..r and every anchor; anchor i sees every document
    token and anchors 0..i."""
    N = n_doc + n_slot
    m = np.zeros((N, N), dtype=bool)
    for r in range(n_doc):
        m[r, :r + 1] = True
        m[r, n_doc:] = True
    for i in range(n_slot):
        row = n_doc + i
        m[row, :n_doc] = True
        m[row, n_doc:n_doc + i + 1] = True
    return m


def extraction_positions(n_doc: int, n_slot: int, k: int) -> np.ndarray:
    """Documents at 0..n_doc-1, slot i at the last token of its block."""
    doc = list(range(n_doc))
    slots = [extraction_slot_position(i, n_doc, k) for i in range(n_slot)]
    return np.asarray(doc + slots, dtype=np.int64)


def masked_extraction_attention(q_pre, k_pre, v, n_doc, n_slot, k, theta, rows=None,
                                mask="structured"):
    """Attention over one document and its slots under the structured mask
    (mask="structured") or the anchor-token mask of the ablation
    (mask="anchor", reading S16; the extra tokens take the slots' positions).

    q_pre bits [N][Hq][d], k_pre/v bits [N][Hkv][d] for the N = n_doc+n_slot
    tokens (pre-RoPE).  q and k are rotated at extraction_positions() in fp64
    (no rounding).  Returns out fp64 [N][Hq][d], or [len(rows)][Hq][d] for
    the query rows listed in `rows` (each row computed exactly as in the full
    result)."""
    N, hq, d = q_pre.shape
    hkv = k_pre.shape[1]
    g = hq // hkv
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    pos = extraction_positions(n_doc, n_slot, k)
    q = rope_rotate(bf16_to_f64(q_pre[rows]).transpose(1, 0, 2), pos[rows], theta)
    kk = rope_rotate(bf16_to_f64(k_pre).transpose(1, 0, 2), pos, theta)
    vv = bf16_to_f64(v).transpose(1, 0, 2)
    if mask == "structured":
        vis = structured_mask(n_doc, n_slot, k)[rows]
    elif mask == "anchor":
        vis = anchor_mask(n_doc, n_slot)[rows]
    else:
        raise ValueError("unknown mask %r" % (mask,))
    out = np.empty((len(rows), hq, d), dtype=np.float64)
    for h in range(hq):
        out[:, h, :] = masked_softmax_attention(q[h], kk[h // g], vv[h // g], vis)
    return out


# ---------------------------------------------------------------------------
# Byte accounting
# ---------------------------------------------------------------------------


def kv_bytes_per_slot(n_layers: int, n_kv_heads: int, head_dim: int,
                      elem_bytes: int = 2) -> int:
    """K and V bytes one composed slot occupies over all layers."""
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes
