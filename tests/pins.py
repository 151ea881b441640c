"""Checks that tie the CPU oracle to facts fixed outside the oracle itself.

Each check takes the oracle module and raises AssertionError on a mismatch.
tests/test_oracle_pins.py runs every check against the real oracle and
against copies with a planted mistake (to show each check has teeth).
Sources: the C2KV explainer (paper-daily.com) sections "C2 tokens",
"structured information flow" and "positions at concatenation"; the Llama 3
paragraph of the KV-cache essay (feinterview.poetries.top); textbook
identities of rotations and of softmax.
"""
import math

import numpy as np
import torch
from scipy.special import expit

from conftest import read_golden


# --------------------------------------------------------------- positions

def check_blog_positions(o):
    g = read_golden("positions_400tok_k4.txt")
    k = g["k"][0]
    n0, s0 = g["doc0_tokens"][0], g["doc0_slots"][0]
    assert o.slot_count(n0, k) == s0
    pos, l_tot = o.composed_positions([n0, 40], [s0, o.slot_count(40, k)], k)
    want0 = np.arange(g["doc0_first"][0], g["doc0_last"][0] + 1, g["doc0_step"][0])
    assert len(want0) == s0
    assert np.array_equal(pos[:s0], want0), pos[:5]
    assert pos[s0] == g["doc1_first"][0], pos[s0]
    assert l_tot == n0 + 40
    e = g["extraction_first_slots"]
    assert [o.extraction_slot_position(j, n0, k) for j in range(len(e))] == e


def check_slot_counts(o):
    for n, k, s in read_golden("slot_counts.txt")["_rows"]:
        assert o.slot_count(n, k) == s, (n, k)


def _brute_positions(docs, k):
    """Lay the original text out token by token and read each slot's position
    off the last token of its block (independent of the oracle's formula)."""
    out = []
    cursor = 0
    for n, s in docs:
        global_pos = list(range(cursor, cursor + n))
        blocks = {}
        for t in range(n):
            blocks[t // k] = global_pos[t]      # later tokens overwrite: last one wins
        for j in range(s):
            out.append(blocks[j])
        cursor += n
    return out


def check_positions_bruteforce(o):
    rng = np.random.default_rng(7)
    for trial in range(40):
        k = int(rng.choice([1, 2, 4, 8, 16]))
        ndoc = int(rng.integers(1, 7))
        lens = [int(rng.integers(1, 60)) for _ in range(ndoc)]
        docs = [(n, o.slot_count(n, k)) for n in lens]
        want = _brute_positions(docs, k)
        assert [len({t // k for t in range(n)}) for n in lens] == [s for _, s in docs]
        ids = list(range(ndoc))
        order = [int(x) for x in rng.permutation(ndoc)]
        seq = o.composed_order(ids, order)
        assert seq == order
        pos, l_tot = o.composed_positions([docs[i][0] for i in seq],
                                          [docs[i][1] for i in seq], k)
        assert pos.tolist() == _brute_positions([docs[i] for i in seq], k)
        assert l_tot == sum(lens)
        pos_id, _ = o.composed_positions(lens, [s for _, s in docs], k)
        assert pos_id.tolist() == want


# ------------------------------------------------------------------ mask

def check_no_realign_positions(o):
    """The "no position re-alignment" ablation (section "results", reading
    S15): every document keeps the positions it was extracted at.  With the
    worked example's 400-token document followed by a 40-token one, the second
    document's slots restart at the extraction positions 3, 7, ... instead of
    403; the question still starts after both documents' original length.
    Also brute force: each document laid out alone from position 0."""
    g = read_golden("positions_400tok_k4.txt")
    k = g["k"][0]
    n0, s0 = g["doc0_tokens"][0], g["doc0_slots"][0]
    s1 = o.slot_count(40, k)
    pos, l_tot = o.composed_positions([n0, 40], [s0, s1], k, realign=False)
    want0 = np.arange(g["doc0_first"][0], g["doc0_last"][0] + 1, g["doc0_step"][0])
    assert np.array_equal(pos[:s0], want0)
    e = g["extraction_first_slots"]
    assert list(pos[s0:s0 + len(e)]) == e, pos[s0:s0 + 4]
    assert pos[s0] != g["doc1_first"][0]
    assert l_tot == n0 + 40
    rng = np.random.default_rng(11)
    for _ in range(20):
        kk = int(rng.integers(1, 9))
        docs = []
        for _ in range(int(rng.integers(1, 5))):
            n = int(rng.integers(1, 60))
            docs.append((n, -(-n // kk)))
        brute = []
        for n, s in docs:
            brute += _brute_positions([(n, s)], kk)   # each document alone, from 0
        got, lt = o.composed_positions([d[0] for d in docs], [d[1] for d in docs], kk, realign=False)
        assert list(got) == brute and lt == sum(d[0] for d in docs)


def check_blog_mask(o):
    g = read_golden("structured_mask_k4_12tok_3slot.txt")
    k, n, m = g["k"][0], g["n_doc"][0], g["n_slot"][0]
    M = o.structured_mask(n, m, k)
    assert M.shape == (n + m, n + m)
    slot_doc = M[n:, :n]
    assert int(slot_doc.sum()) == g["c2kv_slot_doc_cells"][0]
    assert m * n == g["plain_causal_slot_doc_cells"][0]
    for i in range(m):
        seen = [c + 1 for c in range(n) if slot_doc[i, c]]
        assert seen == g["slot%d" % (i + 1)], (i, seen)
    assert not M[:n, n:].any()                      # documents never see slots
    assert np.array_equal(M[:n, :n], np.tril(np.ones((n, n), bool)))
    assert np.array_equal(M[n:, n:], np.tril(np.ones((m, m), bool)))
    assert int(M.sum()) == n * (n + 1) // 2 + 20 + m * (m + 1) // 2


def check_extraction_positions(o):
    g = read_golden("positions_400tok_k4.txt")
    p = o.extraction_positions(12, 3, 4)
    assert p[:12].tolist() == list(range(12))
    assert p[12:14].tolist() == g["extraction_first_slots"]
    assert p[14] == 11


# ------------------------------------------------------------------ bf16

def check_bf16_conversion(o):
    rng = np.random.default_rng(3)
    x32 = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormals
        (rng.standard_normal(2000) * 1e38).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.4e38], np.float32),
    ])
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = o.f64_to_bf16(x32.astype(np.float64))
    assert np.array_equal(got, ref)
    # ties to even, and no double rounding through fp32
    one = 1.0
    assert o.f64_to_bf16(np.array([one + 2.0 ** -8]))[0] == 0x3F80
    assert o.f64_to_bf16(np.array([one + 3 * 2.0 ** -8]))[0] == 0x3F82
    assert o.f64_to_bf16(np.array([one + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert o.f64_to_bf16(np.array([np.inf, -np.inf]))[0] == 0x7F80
    bits = rng.integers(0, 0x7F80, 5000).astype(np.uint16)
    assert np.array_equal(o.f64_to_bf16(o.bf16_to_f64(bits)), bits)
    assert o.bf16_to_f64(np.array([0x3F80, 0xC000], np.uint16)).tolist() == [1.0, -2.0]


# ------------------------------------------------------------------ RoPE

def check_rope(o):
    rng = np.random.default_rng(11)
    d, theta = 8, 1.0e4
    inv = o.rope_inv_freq(theta, d)
    assert inv[0] == 1.0
    assert np.allclose(inv[1:] / inv[:-1], theta ** (-2.0 / d), rtol=1e-14)
    x = rng.standard_normal((3, 5, d))
    assert np.array_equal(o.rope_rotate(x, np.zeros(5, np.int64), theta), x)
    pos = rng.integers(0, 200000, 5)
    y = o.rope_rotate(x, pos, theta)
    # rotate-half pairing (i, i+d/2) equals multiplying z_i = x_i + 1j x_{i+d/2}
    # by exp(1j * pos * inv_freq_i)
    h = d // 2
    z = (x[..., :h] + 1j * x[..., h:]) * np.exp(1j * pos[:, None] * inv[None, :])
    assert np.allclose(y[..., :h], z.real, atol=1e-9)
    assert np.allclose(y[..., h:], z.imag, atol=1e-9)
    # composition of rotations, and the relative-position property
    a, b = rng.integers(0, 5000, 5), rng.integers(0, 5000, 5)
    assert np.allclose(o.rope_rotate(o.rope_rotate(x, a, theta), b, theta),
                       o.rope_rotate(x, a + b, theta), atol=1e-9)
    q, kk = rng.standard_normal(d), rng.standard_normal(d)
    dots = []
    for shift in (0, 17, 123456):
        pq = np.array([shift + 40]); pk = np.array([shift + 3])
        dots.append(float(o.rope_rotate(q[None], pq, theta)[0] @ o.rope_rotate(kk[None], pk, theta)[0]))
    assert np.allclose(dots, dots[0], atol=1e-9)


# ------------------------------------------------------------- attention

def _bits(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def check_attention_special_cases(o):
    rng = np.random.default_rng(5)
    d = 16
    q = rng.standard_normal((3, d))
    V = rng.standard_normal((6, d))
    K = rng.standard_normal((6, d))
    # one visible key -> its value
    mask = np.zeros((3, 6), bool); mask[:, 2] = True
    assert np.allclose(o.masked_softmax_attention(q, K, V, mask), V[[2, 2, 2]])
    # identical keys -> mean of the values
    Ks = np.repeat(K[:1], 6, axis=0)
    full = np.ones((3, 6), bool)
    assert np.allclose(o.masked_softmax_attention(q, Ks, V, full), V.mean(0)[None].repeat(3, 0))
    # two keys: closed form through the logistic function, scale 1/sqrt(d)
    a, b = 1.7, -0.4
    q1 = np.zeros((1, d)); q1[0, 0] = 1.0
    K2 = np.zeros((2, d)); K2[0, 0] = a; K2[1, 0] = b
    V2 = rng.standard_normal((2, d))
    w = expit((a - b) / math.sqrt(d))
    want = V2[1] + w * (V2[0] - V2[1])
    assert np.allclose(o.masked_softmax_attention(q1, K2, V2, np.ones((1, 2), bool))[0], want)
    # one dominant logit -> that value
    Kd = K.copy(); Kd[4] = q[0] * 400.0
    out = o.masked_softmax_attention(q[:1], Kd, V, np.ones((1, 6), bool))
    assert np.allclose(out[0], V[4], atol=1e-9)
    # convex combination, invariant to a permutation of the keys
    out = o.masked_softmax_attention(q, K, V, full)
    assert np.all(out <= V.max(0) + 1e-12) and np.all(out >= V.min(0) - 1e-12)
    perm = rng.permutation(6)
    assert np.allclose(o.masked_softmax_attention(q, K[perm], V[perm], full), out)


def check_gqa_and_causality(o):
    rng = np.random.default_rng(9)
    hq, hkv, d, n, t, theta = 6, 2, 16, 7, 4, 1.0e4
    g = hq // hkv
    q = _bits(rng, (t, hq, d)); kn = _bits(rng, (t, hkv, d))
    kc = _bits(rng, (hkv, n, d))
    # every value of kv head j is the constant j+1 -> output head h reads h//g + 1
    vc = np.zeros((hkv, n, d), np.uint16); vn = np.zeros((t, hkv, d), np.uint16)
    for j in range(hkv):
        c = o.f64_to_bf16(np.array([j + 1.0]))[0]
        vc[j] = c; vn[:, j] = c
    out, _ = o.attend_new_tokens(q, kn, vn, kc, vc, 1000, theta)
    for h in range(hq):
        assert np.allclose(out[:, h, :], h // g + 1), h
    # causal: changing new token 3 leaves rows 0..2 unchanged, changes row 3
    vr = _bits(rng, (hkv, n, d)); vnr = _bits(rng, (t, hkv, d))
    o1, _ = o.attend_new_tokens(q, kn, vnr, kc, vr, 50, theta)
    vn2 = vnr.copy(); vn2[3] = _bits(rng, (hkv, d))
    kn2 = kn.copy(); kn2[3] = _bits(rng, (hkv, d))
    o2, _ = o.attend_new_tokens(q, kn2, vn2, kc, vr, 50, theta)
    assert np.array_equal(o1[:3], o2[:3])
    assert not np.allclose(o1[3], o2[3])
    # a decode step is the last row of the same tokens prefilled together
    od, _, _ = o.decode_sequence(q, kn, vnr, kc, vr, 50, theta)
    assert np.allclose(od, o1, atol=1e-12)


def check_k1_equals_uncompressed(o):
    """k=1: every token is its own slot, so the composed cache must be the
    plain RoPE cache of the concatenated documents at positions 0..L_tot-1."""
    rng = np.random.default_rng(13)
    L, hkv, d, theta = 2, 2, 16, 5.0e5
    lens = [5, 1, 9, 3]
    store = {}
    for i, n in enumerate(lens):
        store[10 + i] = (n, n, _bits(rng, (L, hkv, n, d)), _bits(rng, (L, hkv, n, d)))
    ids = [10, 11, 12, 13]
    order = [2, 0, 3, 1]
    pos, l_tot, krot, vcat = o.compose(store, ids, order, 1, theta)
    seq = [ids[i] for i in order]
    raw_k = np.concatenate([store[s][2] for s in seq], axis=2)
    raw_v = np.concatenate([store[s][3] for s in seq], axis=2)
    assert pos.tolist() == list(range(sum(lens))) and l_tot == sum(lens)
    x = o.bf16_to_f64(raw_k)
    want = np.empty_like(x)
    inv = o.rope_inv_freq(theta, d)
    for p in range(l_tot):   # rotate token by token via complex numbers
        h = d // 2
        z = (x[..., p, :h] + 1j * x[..., p, h:]) * np.exp(1j * p * inv)
        want[..., p, :h], want[..., p, h:] = z.real, z.imag
    assert np.all(o.bf16_ulp_distance(krot, o.f64_to_bf16(want)) <= 1)
    assert np.array_equal(vcat, raw_v)


def check_empty_composition(o):
    """A request of no documents composes the concatenation of no segments: no
    positions, L_tot = 0, K and V of 0 rows with the store's geometry; and a
    request of one document is that document alone at positions from 0."""
    rng = np.random.default_rng(17)
    L, hkv, d, theta = 2, 3, 8, 1.0e4
    store = {7: (12, 3, _bits(rng, (L, hkv, 3, d)), _bits(rng, (L, hkv, 3, d)))}
    pos, l_tot, krot, vcat = o.compose(store, [], None, 4, theta)
    assert pos.shape == (0,) and l_tot == 0
    assert krot.shape == (L, hkv, 0, d) and vcat.shape == (L, hkv, 0, d)
    pos, l_tot, krot, vcat = o.compose(store, [7], None, 4, theta, layers=[1])
    assert pos.tolist() == [3, 7, 11] and l_tot == 12
    assert krot.shape == (1, hkv, 3, d) and np.array_equal(vcat[0], store[7][3][1])


def check_k1_attention_equals_uncompressed(o):
    """k=1 (section "C2 tokens": one slot per k tokens, so every token is its
    own slot): composing the documents, prefilling the question after them and
    decoding the answer must be exactly the causal attention of the plain,
    uncompressed token sequence, with token t at position t for every t < L_tot
    + Q + T (section "positions at concatenation": documents keep their
    original lengths of positions, the question follows them).  The reference
    is torch's fp64 scaled_dot_product_attention (a library routine) over
    keys rotated token by token through complex multiplication at arange
    positions and rounded to bf16 as the cache stores them; it shares neither
    the oracle's position bookkeeping nor its attention."""
    rng = np.random.default_rng(23)
    hq, hkv, d, theta = 4, 2, 16, 5.0e5
    lens = [6, 2, 5]
    ids = [20, 21, 22]
    order = [1, 2, 0]
    store = {i: (n, n, _bits(rng, (1, hkv, n, d)), _bits(rng, (1, hkv, n, d))) for i, n in zip(ids, lens)}
    Q, T = 3, 4
    q, kn, vn = _bits(rng, (Q + T, hq, d)), _bits(rng, (Q + T, hkv, d)), _bits(rng, (Q + T, hkv, d))
    # the oracle's path: compose at k=1, the question at L_tot, decode after it
    _, l_tot, kc, vc = o.compose(store, ids, order, 1, theta)
    kc, vc = kc[0], vc[0]
    out_q, kq = o.attend_new_tokens(q[:Q], kn[:Q], vn[:Q], kc, vc, l_tot, theta)
    kc = np.concatenate([kc, kq], axis=1)
    vc = np.concatenate([vc, vn[:Q].transpose(1, 0, 2)], axis=1)
    out_d, _, _ = o.decode_sequence(q[Q:], kn[Q:], vn[Q:], kc, vc, l_tot + Q, theta)
    got = np.concatenate([out_q, out_d], axis=0)                 # [Q+T][hq][d]
    # the reference: the token sequence written out, position = index
    seq = [ids[i] for i in order]
    k_all = np.concatenate([store[s][2][0] for s in seq] + [kn.transpose(1, 0, 2)], axis=1)
    v_all = np.concatenate([store[s][3][0] for s in seq] + [vn.transpose(1, 0, 2)], axis=1)
    n_all = k_all.shape[1]
    assert n_all == sum(lens) + Q + T
    inv = np.power(theta, -2.0 * np.arange(d // 2) / d)

    def rot(x, p):   # x [..., n, d] fp64 at positions p[n]
        z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * p[:, None] * inv[None, :])
        return np.concatenate([z.real, z.imag], axis=-1)

    t_all = np.arange(n_all, dtype=np.float64)
    kr = o.bf16_to_f64(o.f64_to_bf16(rot(o.bf16_to_f64(k_all), t_all)))   # stored as bf16
    qr = rot(o.bf16_to_f64(q).transpose(1, 0, 2), t_all[sum(lens):])      # q is not rounded
    vis = np.arange(n_all)[None, :] <= np.arange(sum(lens), n_all)[:, None]
    g = hq // hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr), torch.from_numpy(np.repeat(kr, g, axis=0)),
        torch.from_numpy(np.repeat(o.bf16_to_f64(v_all), g, axis=0)),
        attn_mask=torch.from_numpy(vis)).numpy().transpose(1, 0, 2)
    assert np.allclose(got, ref, rtol=0, atol=1e-12), np.abs(got - ref).max()


def check_ulp_distance(o):
    """bf16_ulp_distance, the comparator of every re-rotated key, against its
    definition: the number of steps between two values along the ordered set
    of distinct finite bf16 values (+0 and -0 are one value).  The ordered set
    is built here from torch's bf16 -> fp64 widening (a library routine), and
    hand pairs cover +-0, neighbours, a 2-ulp gap, a binade edge, the sign
    boundary and the largest finite values."""
    allbits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).double().numpy()
    finite = np.isfinite(vals)
    distinct = np.unique(vals[finite])            # sorted; -0 and +0 compare equal
    rank = np.full(0x10000, -1, np.int64)
    rank[finite] = np.searchsorted(distinct, vals[finite])
    hand = [(0x3F80, 0x3F80, 0), (0x3F80, 0x3F81, 1), (0x3F80, 0x3F82, 2), (0x3F7F, 0x3F80, 1),
            (0x0000, 0x8000, 0), (0x0001, 0x8001, 2), (0x0001, 0x0000, 1), (0xBF80, 0xBF81, 1),
            (0x3F80, 0x4000, 128), (0x7F7F, 0x7F7E, 1), (0x7F7F, 0xFF7F, int(rank[0x7F7F] - rank[0xFF7F]))]
    for a, b, want in hand:
        assert int(rank[b] - rank[a]) in (want, -want), (hex(a), hex(b))
        got = o.bf16_ulp_distance(np.array([a], np.uint16), np.array([b], np.uint16))
        assert int(got[0]) == want, (hex(a), hex(b), int(got[0]), want)
    rng = np.random.default_rng(31)
    fin = allbits[finite]
    a = rng.choice(fin, 20000)
    near = np.clip(rank[a] + rng.integers(-3, 4, a.size), 0, distinct.size - 1)
    # b: half random finite values, half within 3 steps of a (a bit pattern of that value)
    first_of = np.full(distinct.size, 0, np.int64)
    first_of[rank[fin][::-1]] = fin[::-1]
    b = np.where(rng.random(a.size) < 0.5, rng.choice(fin, a.size), first_of[near]).astype(np.uint16)
    want = np.abs(rank[a] - rank[b])
    assert np.array_equal(o.bf16_ulp_distance(a, b), want)


def check_llama3_bytes(o):
    g = read_golden("kv_bytes_llama3.txt")
    assert o.kv_bytes_per_slot(g["n_layers"][0], g["n_kv_heads"][0],
                               g["head_dim"][0]) == g["bytes_per_token"][0]


def check_structured_attention_on_the_blog_figure(o):
    """The k=4 figure of section "structured information flow" (12 document
    tokens, 3 slots), run through the whole extraction attention: with q = 0
    every score is 0, so each row is the plain mean of the values it sees,
    and value j = e_j shows exactly which keys.  Slot rows must see the
    document cells the figure lists and the slots up to themselves; document
    rows their causal prefix and no slot."""
    g = read_golden("structured_mask_k4_12tok_3slot.txt")
    k, n, m = g["k"][0], g["n_doc"][0], g["n_slot"][0]
    N, d = n + m, 16
    rng = np.random.default_rng(29)
    q = np.zeros((N, 2, d), np.uint16)
    kk = _bits(rng, (N, 1, d))
    one = o.f64_to_bf16(np.array([1.0]))[0]
    v = np.zeros((N, 1, d), np.uint16)
    for j in range(N):
        v[j, 0, j] = one
    out = o.masked_extraction_attention(q, kk, v, n, m, k, 1.0e4, mask="structured")
    for r in range(N):
        if r < n:
            seen = set(range(r + 1))
        else:
            i = r - n
            seen = {c - 1 for c in g["slot%d" % (i + 1)]} | set(range(n, r + 1))
        want = np.zeros(d)
        want[sorted(seen)] = 1.0 / len(seen)
        for h in range(2):
            assert np.allclose(out[r, h], want, atol=1e-12), (r, h)


# ----------------------------------------------------- anchor-token ablation

def check_anchor_mask_uniform_scores(o):
    """Anchor-token ablation (section "results"): the extra tokens and the
    document tokens see each other in both directions, so the document
    tokens' outputs are rewritten by the anchors.  With q = 0 every score is
    0 and each output row is the plain mean of the values it can see; with
    value j the unit vector e_j the row shows exactly which keys it saw.
    Expected: document token r sees documents 0..r (the base causal mask is
    kept among the documents) and every anchor; anchor i sees every document
    token and anchors 0..i."""
    rng = np.random.default_rng(17)
    n_doc, k, d, theta = 7, 3, 16, 1.0e4
    n_slot = -(-n_doc // k)
    N = n_doc + n_slot
    q = np.zeros((N, 2, d), np.uint16)
    kk = _bits(rng, (N, 1, d))
    one = o.f64_to_bf16(np.array([1.0]))[0]
    v = np.zeros((N, 1, d), np.uint16)
    for j in range(N):
        v[j, 0, j] = one
    out = o.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, theta, mask="anchor")
    for r in range(N):
        if r < n_doc:
            seen = set(range(r + 1)) | set(range(n_doc, N))
        else:
            seen = set(range(n_doc)) | set(range(n_doc, r + 1))
        want = np.zeros(d)
        want[sorted(seen)] = 1.0 / len(seen)
        for h in range(2):
            assert np.allclose(out[r, h], want, atol=1e-12), (r, h)
    # the structured mask on the same input: documents see no anchor
    st = o.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, theta, mask="structured")
    assert np.allclose(st[0, 0, :N], np.eye(N)[0], atol=1e-12)


def check_anchor_rows_are_causal_attention(o):
    """Anchor rows see every earlier token of the sequence, so they are plain
    causal attention (torch's fp64 scaled_dot_product_attention) over the
    sequence rotated at its extraction positions; with no anchors the whole
    result is causal attention at positions 0..n-1."""
    rng = np.random.default_rng(19)
    hq, hkv, d, theta = 4, 2, 16, 5.0e5
    for n_doc, k in ((9, 4), (5, 1), (6, 0)):
        n_slot = -(-n_doc // k) if k else 0
        kk_ = max(k, 1)
        N = n_doc + n_slot
        q, kk, v = _bits(rng, (N, hq, d)), _bits(rng, (N, hkv, d)), _bits(rng, (N, hkv, d))
        out = o.masked_extraction_attention(q, kk, v, n_doc, n_slot, kk_, theta, mask="anchor")
        pos = o.extraction_positions(n_doc, n_slot, kk_)
        qr = o.rope_rotate(o.bf16_to_f64(q).transpose(1, 0, 2), pos, theta)
        kr = o.rope_rotate(o.bf16_to_f64(kk).transpose(1, 0, 2), pos, theta)
        vr = o.bf16_to_f64(v).transpose(1, 0, 2)
        g = hq // hkv
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qr), torch.from_numpy(np.repeat(kr, g, axis=0)),
            torch.from_numpy(np.repeat(vr, g, axis=0)), is_causal=True).numpy().transpose(1, 0, 2)
        rows = slice(n_doc, N) if n_slot else slice(0, N)
        assert np.allclose(out[rows], ref[rows], atol=1e-12), (n_doc, k)
        if n_slot:   # documents that see anchors are not causal rows
            assert not np.allclose(out[:n_doc - 1], ref[:n_doc - 1], atol=1e-6)


ALL_CHECKS = [
    check_blog_positions, check_slot_counts, check_positions_bruteforce, check_no_realign_positions,
    check_blog_mask, check_extraction_positions, check_bf16_conversion,
    check_rope, check_attention_special_cases, check_gqa_and_causality,
    check_k1_equals_uncompressed, check_empty_composition, check_k1_attention_equals_uncompressed,
    check_ulp_distance,
    check_llama3_bytes,
    check_structured_attention_on_the_blog_figure,
    check_anchor_mask_uniform_scores, check_anchor_rows_are_causal_attention,
]


# ------------------------------------------------- decoder step (D17 reading)

def check_rms_norm(d):
    """RMSNorm against its definition written as a loop, and a closed form:
    a constant row c gives c / sqrt(c^2 + eps) times the weights."""
    rng = np.random.default_rng(41)
    eps = 1e-5
    x = _bits(rng, (3, 24))
    w = _bits(rng, (24,))
    got = d.rms_norm(x, w, eps)
    xf, wf = d.O.bf16_to_f64(x), d.O.bf16_to_f64(w)
    for t in range(3):
        ss = 0.0
        for i in range(24):
            ss += xf[t, i] * xf[t, i]
        r = math.sqrt(ss / 24 + eps)
        for i in range(24):
            assert abs(got[t, i] - xf[t, i] / r * wf[i]) <= 1e-12 * (1 + abs(got[t, i]))
    c = 0.375
    xc = np.full((1, 16), d.O.f64_to_bf16(np.array([c]))[0], np.uint16)
    assert np.allclose(d.rms_norm(xc, w[:16], eps)[0], c / math.sqrt(c * c + eps) * wf[:16], rtol=1e-12)


def check_linear(d):
    """x W^T against the triple loop."""
    rng = np.random.default_rng(43)
    x, w = _bits(rng, (3, 20)), _bits(rng, (7, 20))
    got = d.linear(x, w)
    xf, wf = d.O.bf16_to_f64(x), d.O.bf16_to_f64(w)
    for t in range(3):
        for n in range(7):
            acc = 0.0
            for k in range(20):
                acc += xf[t, k] * wf[n, k]
            assert abs(got[t, n] - acc) <= 1e-12 * (1 + abs(acc))


def check_silu_and_gate_up_layout(d):
    """silu(g) = g * sigmoid(g) (scipy's expit, a library routine), 0 at 0;
    and the fused gate/up weight in the library's layout (64-row gate and up
    blocks per 128-row tile) gives silu(h W_g^T) * (h W_u^T) of the separate
    weights."""
    g = np.linspace(-30, 30, 601)
    assert np.allclose(d.silu(g), g * expit(g), rtol=1e-13, atol=1e-300)
    assert d.silu(np.array([0.0]))[0] == 0.0
    rng = np.random.default_rng(47)
    F, k = 192, 32
    wg, wu = _bits(rng, (F, k)), _bits(rng, (F, k))
    fused = np.empty((2 * F, k), np.uint16)
    for i in range(F // 64):
        fused[128 * i:128 * i + 64] = wg[64 * i:64 * i + 64]
        fused[128 * i + 64:128 * i + 128] = wu[64 * i:64 * i + 64]
    h = _bits(rng, (2, k))
    hf = d.O.bf16_to_f64(h)
    gate = hf @ d.O.bf16_to_f64(wg).T
    up = hf @ d.O.bf16_to_f64(wu).T
    assert np.allclose(d.swiglu(h, fused), gate * expit(gate) * up, rtol=1e-12)


def _decoder_case(d, rng, zero=()):
    B, Hq, Hkv, hd, n, F = 2, 4, 2, 16, 9, 128
    dim = Hq * hd
    w = {"attn_norm": _bits(rng, (dim,)), "mlp_norm": _bits(rng, (dim,)),
         "qkv": _bits(rng, ((Hq + 2 * Hkv) * hd, dim), 0.2), "o": _bits(rng, (dim, Hq * hd), 0.2),
         "gate_up": _bits(rng, (2 * F, dim), 0.2), "down": _bits(rng, (dim, F), 0.2)}
    for name in zero:
        w[name] = np.zeros_like(w[name])
    x = _bits(rng, (B, dim))
    kc = [_bits(rng, (Hkv, n, hd)) for _ in range(B)]
    vc = [_bits(rng, (Hkv, n, hd)) for _ in range(B)]
    return x, w, kc, vc, (Hq, Hkv, hd)


def check_decoder_layer_residuals_and_attention(d):
    """A layer whose output projections are zero is the identity on the
    residual stream; with q = 0 (zero q rows of the QKV weight) every key
    scores the same, so each head's attention output is the plain mean of
    its kv head's cached values and the new token's value."""
    rng = np.random.default_rng(53)
    x, w, kc, vc, (Hq, Hkv, hd) = _decoder_case(d, rng, zero=("o", "down"))
    x2, st = d.decoder_layer_decode(x, w, kc, vc, [20, 31], 1.0e4, Hq, Hkv, 1e-5)
    assert np.array_equal(x2, x) and np.array_equal(st["x1"], x)
    x, w, kc, vc, (Hq, Hkv, hd) = _decoder_case(d, rng)
    w["qkv"][:Hq * hd] = 0
    x2, st = d.decoder_layer_decode(x, w, kc, vc, [20, 31], 1.0e4, Hq, Hkv, 1e-5)
    G = Hq // Hkv
    for b in range(2):
        vnew = d.O.bf16_to_f64(st["v"][b].reshape(Hkv, hd))
        for h in range(Hq):
            vals = np.concatenate([d.O.bf16_to_f64(vc[b][h // G]), vnew[h // G][None]], axis=0)
            want = d.O.f64_to_bf16(vals.mean(axis=0))
            assert np.array_equal(st["att"][b].reshape(Hq, hd)[h], want), (b, h)
    # the layer's output differs from its input once the projections are live
    assert not np.array_equal(x2, x)


# checks of the decoder-step oracle (they take oracle.decoder_oracle)
DECODER_CHECKS = [check_rms_norm, check_linear, check_silu_and_gate_up_layout,
                  check_decoder_layer_residuals_and_attention]
