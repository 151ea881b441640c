"""The CPU oracle against its pins, and each pin against a planted mistake.

A planted mistake is a plausible bug put into the oracle on the CPU (via
monkeypatch, undone after the test); the matching pin must then fail.
"""
import numpy as np
import pytest

import oracle.c2kv_oracle as O
import oracle.decoder_oracle as DO
import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(O)


@pytest.mark.parametrize("check", pins.DECODER_CHECKS, ids=lambda c: c.__name__)
def test_decoder_pin(check):
    check(DO)


def _rms_no_eps(x_bits, w_bits, eps):
    x = O.bf16_to_f64(x_bits)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) * O.bf16_to_f64(w_bits)[None, :]


def _rms_sum_not_mean(x_bits, w_bits, eps):
    x = O.bf16_to_f64(x_bits)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps) * O.bf16_to_f64(w_bits)[None, :]


def _linear_last_column_dropped(x_bits, w_bits):
    return O.bf16_to_f64(x_bits)[:, :-1] @ O.bf16_to_f64(w_bits)[:, :-1].T


def _silu_as_sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


def _gate_up_swapped(w_gu_bits):
    n2, k = w_gu_bits.shape
    blocks = w_gu_bits.reshape(n2 // 128, 2, 64, k)
    return blocks[:, 1].reshape(-1, k), blocks[:, 0].reshape(-1, k)


_REAL_LAYER = DO.decoder_layer_decode


def _layer_without_mlp_residual(x_bits, w, k_caches, v_caches, start_pos, theta, hq, hkv, eps):
    x2, st = _REAL_LAYER(x_bits, w, k_caches, v_caches, start_pos, theta, hq, hkv, eps)
    m_out = DO.linear(st["m"], w["down"])
    return DO.bf16(m_out), st


DECODER_MUTATIONS = [
    ("rms_norm", _rms_no_eps, pins.check_rms_norm),
    ("rms_norm", _rms_sum_not_mean, pins.check_rms_norm),
    ("linear", _linear_last_column_dropped, pins.check_linear),
    ("silu", _silu_as_sigmoid, pins.check_silu_and_gate_up_layout),
    ("split_gate_up", _gate_up_swapped, pins.check_silu_and_gate_up_layout),
    ("decoder_layer_decode", _layer_without_mlp_residual, pins.check_decoder_layer_residuals_and_attention),
]


@pytest.mark.parametrize("name,bad,check", DECODER_MUTATIONS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in DECODER_MUTATIONS])
def test_decoder_planted_mistake_is_caught(monkeypatch, name, bad, check):
    monkeypatch.setattr(DO, name, bad)
    with pytest.raises(AssertionError):
        check(DO)


def test_decoder_attention_position_mistake_is_caught(monkeypatch):
    """The decoder step's attention goes through attend_new_tokens: a GQA
    mapping mistake there (h % G) breaks the q = 0 mean check of the layer."""
    real = O.attend_new_tokens

    def modulo_mapping(q_pre, k_new_pre, v_new, k_cache, v_cache, start_pos, theta):
        t, hq, dd = q_pre.shape
        hkv = k_new_pre.shape[1]
        out, kr = real(q_pre, k_new_pre, v_new, k_cache, v_cache, start_pos, theta)
        perm = [h % hkv * (hq // hkv) + h // hkv for h in range(hq)]
        return out[:, perm], kr

    monkeypatch.setattr(O, "attend_new_tokens", modulo_mapping)
    with pytest.raises(AssertionError):
        pins.check_decoder_layer_residuals_and_attention(DO)


def _positions_no_minus_one(n_tokens, n_slots, k, realign=True):
    pos, off = [], 0
    for n, s in zip(n_tokens, n_slots):
        pos += [(off if realign else 0) + min((j + 1) * k, n) for j in range(s)]
        off += n
    return np.asarray(pos, np.int64), off


def _positions_offset_by_slots(n_tokens, n_slots, k, realign=True):
    pos, off = [], 0
    for n, s in zip(n_tokens, n_slots):
        pos += [(off if realign else 0) + min((j + 1) * k, n) - 1 for j in range(s)]
        off += s
    return np.asarray(pos, np.int64), off


def _positions_realign_ignored(n_tokens, n_slots, k, realign=True):
    pos, off = [], 0
    for n, s in zip(n_tokens, n_slots):
        pos += [off + min((j + 1) * k, n) - 1 for j in range(s)]
        off += n
    return np.asarray(pos, np.int64), off


def _positions_no_realign_question_at_slots(n_tokens, n_slots, k, realign=True):
    pos, off = [], 0
    for n, s in zip(n_tokens, n_slots):
        pos += [(off if realign else 0) + min((j + 1) * k, n) - 1 for j in range(s)]
        off += n
    return np.asarray(pos, np.int64), (off if realign else max(n_tokens))


def _rope_sign_flipped(x, pos, theta):
    d = x.shape[-1]; h = d // 2
    a = np.asarray(pos, np.float64)[:, None] * O.rope_inv_freq(theta, d)[None, :]
    c, s = np.cos(a), np.sin(a)
    return np.concatenate([x[..., :h] * c + x[..., h:] * s,
                           x[..., h:] * c - x[..., :h] * s], axis=-1)


def _rope_interleaved(x, pos, theta):
    d = x.shape[-1]
    a = np.asarray(pos, np.float64)[:, None] * O.rope_inv_freq(theta, d)[None, :]
    c, s = np.cos(a), np.sin(a)
    y = x.copy()
    y[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    y[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return y


def _inv_freq_wrong_exponent(theta, d):
    return np.power(float(theta), -np.arange(d // 2, dtype=np.float64) / d)


def _mask_no_sink(n_doc, n_slot, k):
    m = np.zeros((n_doc + n_slot,) * 2, bool)
    for r in range(n_doc):
        m[r, :r + 1] = True
    for i in range(n_slot):
        m[n_doc + i, i * k:min((i + 1) * k, n_doc)] = True
        m[n_doc + i, n_doc:n_doc + i + 1] = True
    return m


def _mask_block_shifted(n_doc, n_slot, k):
    m = np.zeros((n_doc + n_slot,) * 2, bool)
    for r in range(n_doc):
        m[r, :r + 1] = True
    for i in range(n_slot):
        m[n_doc + i, :min(k, n_doc)] = True
        m[n_doc + i, i * k:min((i + 1) * k + 1, n_doc)] = True
        m[n_doc + i, n_doc:n_doc + i + 1] = True
    return m


def _structured_as_causal(n_doc, n_slot, k):
    return np.tril(np.ones((n_doc + n_slot,) * 2, bool))


def _anchor_docs_causal_over_anchors(n_doc, n_slot):
    m = np.tril(np.ones((n_doc + n_slot,) * 2, bool))
    return m


def _anchor_docs_see_anchors_only(n_doc, n_slot):
    m = np.zeros((n_doc + n_slot,) * 2, bool)
    m[:n_doc, n_doc:] = True
    for r in range(n_doc):
        m[r, r] = True
    for i in range(n_slot):
        m[n_doc + i, :n_doc + i + 1] = True
    return m


def _anchor_anchors_see_all_anchors(n_doc, n_slot):
    N = n_doc + n_slot
    m = np.zeros((N, N), bool)
    for r in range(n_doc):
        m[r, :r + 1] = True
        m[r, n_doc:] = True
    m[n_doc:, :] = True
    return m


def _softmax_no_scale(q, K, V, mask):
    s = np.where(mask, q @ K.T, -np.inf)
    p = np.exp(s - s.max(1, keepdims=True))
    return (p / p.sum(1, keepdims=True)) @ V


def _bf16_truncate(x):
    x = np.asarray(x, np.float64)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _bf16_double_round(x):
    x32 = np.asarray(x, np.float64).astype(np.float32)
    import torch
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _attend_question_shifted(q_pre, k_new_pre, v_new, k_cache, v_cache, start_pos, theta):
    """The new tokens placed one position late (start_pos + 1 + i)."""
    return _REAL_ATTEND(q_pre, k_new_pre, v_new, k_cache, v_cache, start_pos + 1, theta)


_REAL_ATTEND = O.attend_new_tokens


def _ulp_always_zero(a_bits, b_bits):
    return np.zeros(np.broadcast(np.asarray(a_bits), np.asarray(b_bits)).shape, np.int32)


def _ulp_sign_magnitude_ignored(a_bits, b_bits):
    """Bit patterns subtracted as plain integers (wrong across the sign)."""
    return np.abs(np.asarray(a_bits, np.int32) - np.asarray(b_bits, np.int32))


def _ulp_off_by_one_across_zero(a_bits, b_bits):
    """-0 and +0 treated as two values."""
    def ordered(bits):
        v = np.asarray(bits, dtype=np.uint16).astype(np.int32)
        return np.where(v & 0x8000, 0x7FFF - v, v)
    return np.abs(ordered(a_bits) - ordered(b_bits))


MUTATIONS = [
    ("composed_positions", _positions_no_minus_one, pins.check_blog_positions),
    ("composed_positions", _positions_offset_by_slots, pins.check_blog_positions),
    ("composed_positions", _positions_realign_ignored, pins.check_no_realign_positions),
    ("composed_positions", _positions_no_realign_question_at_slots, pins.check_no_realign_positions),
    ("rope_rotate", _rope_sign_flipped, pins.check_rope),
    ("rope_rotate", _rope_interleaved, pins.check_rope),
    ("rope_inv_freq", _inv_freq_wrong_exponent, pins.check_rope),
    ("structured_mask", _mask_no_sink, pins.check_blog_mask),
    ("structured_mask", _mask_block_shifted, pins.check_blog_mask),
    ("masked_softmax_attention", _softmax_no_scale, pins.check_attention_special_cases),
    ("structured_mask", _mask_no_sink, pins.check_structured_attention_on_the_blog_figure),
    ("structured_mask", _mask_block_shifted, pins.check_structured_attention_on_the_blog_figure),
    ("structured_mask", _structured_as_causal, pins.check_structured_attention_on_the_blog_figure),
    ("anchor_mask", _anchor_docs_causal_over_anchors, pins.check_anchor_mask_uniform_scores),
    ("anchor_mask", _anchor_docs_causal_over_anchors, pins.check_anchor_rows_are_causal_attention),
    ("anchor_mask", _anchor_docs_see_anchors_only, pins.check_anchor_mask_uniform_scores),
    ("anchor_mask", _anchor_anchors_see_all_anchors, pins.check_anchor_mask_uniform_scores),
    ("anchor_mask", _anchor_anchors_see_all_anchors, pins.check_anchor_rows_are_causal_attention),
    ("f64_to_bf16", _bf16_truncate, pins.check_bf16_conversion),
    ("f64_to_bf16", _bf16_double_round, pins.check_bf16_conversion),
    ("attend_new_tokens", _attend_question_shifted, pins.check_k1_attention_equals_uncompressed),
    ("bf16_ulp_distance", _ulp_always_zero, pins.check_ulp_distance),
    ("bf16_ulp_distance", _ulp_sign_magnitude_ignored, pins.check_ulp_distance),
    ("bf16_ulp_distance", _ulp_off_by_one_across_zero, pins.check_ulp_distance),
]


@pytest.mark.parametrize("name,bad,check", MUTATIONS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bad, check):
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        check(O)


def test_gqa_mapping_mistake_is_caught(monkeypatch):
    """q head h must read kv head h // G, not h % G."""
    real = O.attend_new_tokens

    def modulo_mapping(q_pre, k_new_pre, v_new, k_cache, v_cache, start_pos, theta):
        t, hq, d = q_pre.shape
        hkv = k_new_pre.shape[1]
        perm = [h % hkv * (hq // hkv) + h // hkv for h in range(hq)]
        out, kr = real(q_pre[:, perm], k_new_pre, v_new, k_cache, v_cache, start_pos, theta)
        inv = np.argsort(perm)
        return out[:, inv], kr

    monkeypatch.setattr(O, "attend_new_tokens", modulo_mapping)
    with pytest.raises(AssertionError):
        pins.check_gqa_and_causality(O)


def test_masked_attention_row_subset_equals_full_rows():
    """The sampled-row form of the extraction attention (used at full size)
    computes each row exactly as the full result does."""
    rng = np.random.default_rng(2)
    n_doc, n_slot, k = 37, 10, 4
    N = n_doc + n_slot
    q = (rng.standard_normal((N, 4, 16)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kk = (rng.standard_normal((N, 2, 16)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    v = (rng.standard_normal((N, 2, 16)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    full = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, 1e4)
    rows = [0, 5, 36, 37, 40, 46]
    sub = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, 1e4, rows=rows)
    assert np.array_equal(sub, full[rows])
