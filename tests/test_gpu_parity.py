"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: positions and composition order bit-exact, values bit-exact, re-rotated
keys within 1 bf16 ulp, attention outputs within max-abs 2e-2 / mean-abs
2e-3 (and mean error under 2 % of the output RMS).
"""
import numpy as np
import pytest
import torch

import oracle.c2kv_oracle as O
import compressed_composable_kv_gb300 as P
from compressed_composable_kv_gb300 import synth as S
from gpu_util import Scenario, check_attention, check_keys, check_request, run_all, to_bits, to_dev, upload

pytestmark = pytest.mark.gpu


def test_tiny_end_to_end():
    w = S.WORKLOADS["tiny"]
    docs, reqs = S.make_requests(w)
    sc = Scenario(w.geom, w.k, [(i, n, s) for i, (n, s) in docs.items()],
                  [(r.doc_ids, r.order) for r in reqs], w.q_len, w.decode_steps, seed=w.seed)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    assert sc.batch.n_slots == [113] and sc.batch.l_tot == [452]
    check_request(sc, inputs, pre, dec, 0, layers=[0], steps=range(w.decode_steps))
    sc.close()


def test_tiny_sharp_softmax():
    """q scaled by 4: a few keys dominate, so errors are not hidden by a flat softmax."""
    w = S.WORKLOADS["tiny"]
    docs, reqs = S.make_requests(w)
    sc = Scenario(w.geom, w.k, [(i, n, s) for i, (n, s) in docs.items()],
                  [([2, 0, 1], None)], w.q_len, 4, seed=w.seed)
    inputs = S.make_step_inputs(w, decode_steps=4, q_scale=4.0)
    pre, dec = run_all(sc, upload(inputs))
    check_request(sc, inputs, pre, dec, 0, layers=[0], steps=range(4))
    sc.close()


def test_no_position_realignment_ablation():
    """C2KV_COMPOSE_NO_REALIGN: every document keeps its extraction positions
    (the "results" ablation); the question and answer still follow L_tot."""
    w = S.WORKLOADS["tiny"]
    docs, reqs = S.make_requests(w)
    sc = Scenario(w.geom, w.k, [(i, n, s) for i, (n, s) in docs.items()],
                  [([1, 0, 2], [2, 0, 1])], w.q_len, 6, seed=w.seed, realign=False)
    inputs = S.make_step_inputs(w, decode_steps=6)
    pre, dec = run_all(sc, upload(inputs))
    pos = sc.batch.pos[0][:sc.batch.n_slots[0]].cpu().numpy()
    assert pos.min() == w.k - 1 and sc.batch.l_tot[0] == 452   # documents restart at 3
    check_request(sc, inputs, pre, dec, 0, layers=[0], steps=range(6))
    sc.close()


@pytest.mark.parametrize("realign", [True, False])
def test_layer_pipelined_compose_matches_one_shot(realign):
    """Composing layer groups one by one (C2KV_COMPOSE_CONTINUE) with the
    question prefill of each group enqueued in between gives the same caches
    and outputs, bit for bit, as one compose followed by the prefill; also
    with the no-re-alignment ablation."""
    g = S.Geometry(8, 16, 4, 128, 5.0e5)
    specs = [(1, 900, 225), (2, 333, 84), (3, 1200, 300)]
    requests = [([3, 1, 2], None), ([2, 3], [1, 0])]
    sc = Scenario(g, 4, specs, requests, q_len=24, decode_steps=0, realign=realign)
    bt = sc.batch
    rng = np.random.default_rng(5)
    q = to_dev(S.normal_bf16(rng, (g.n_layers, 2, 24, g.n_q_heads, g.head_dim)))
    kq = to_dev(S.normal_bf16(rng, (g.n_layers, 2, 24, g.n_kv_heads, g.head_dim)))
    vq = to_dev(S.normal_bf16(rng, (g.n_layers, 2, 24, g.n_kv_heads, g.head_dim)))

    def prefill(layers):
        outs = []
        for l in layers:
            o = torch.empty_like(q[l])
            bt.prefill(l, q[l], kq[l], vq[l], o)
            outs.append(o)
        return outs

    for t in bt.k_caches + bt.v_caches:
        t.fill_(7.0)   # rows past N + Q stay untouched by both runs
    bt.compose()
    ref_out = prefill(range(8))
    torch.cuda.synchronize()
    ref_k = [t.clone() for t in bt.k_caches]
    ref_v = [t.clone() for t in bt.v_caches]
    for t in bt.k_caches + bt.v_caches:
        t.fill_(7.0)
    outs = []
    for l0 in range(0, 8, 2):
        bt.compose_layers(l0, l0 + 2)
        outs += prefill(range(l0, l0 + 2))
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    for b in range(2):
        assert torch.equal(bt.k_caches[b], ref_k[b]) and torch.equal(bt.v_caches[b], ref_v[b])
    for l in range(8):
        assert torch.equal(outs[l], ref_out[l])
    # a continuation must follow a composition of the same request into the same table
    other = torch.empty_like(bt.rope_tables[0])
    with pytest.raises(P.C2KVError):
        P.c2kv_compose_layers(sc.store, [3, 1, 2], None, 4, P.C2KV_COMPOSE_CONTINUE, 2, 4, bt.k_caches[0],
                              bt.v_caches[0], bt.cap, other)
    with pytest.raises(P.C2KVError):
        P.c2kv_compose_layers(sc.store, [3, 2, 1], None, 4, P.C2KV_COMPOSE_CONTINUE, 2, 4, bt.k_caches[0],
                              bt.v_caches[0], bt.cap, bt.rope_tables[0])
    with pytest.raises(P.C2KVError):
        P.c2kv_compose_layers(sc.store, [3, 1, 2], None, 4, 0, 4, 4, bt.k_caches[0], bt.v_caches[0], bt.cap,
                              bt.rope_tables[0])
    if not realign:   # a continuation keeps the ablation flag of the composition it continues
        with pytest.raises(P.C2KVError):
            P.c2kv_compose_layers(sc.store, [3, 1, 2], None, 4, P.C2KV_COMPOSE_CONTINUE, 2, 4, bt.k_caches[0],
                                  bt.v_caches[0], bt.cap, bt.rope_tables[0])
    sc.close()


def test_empty_composition_question_only():
    """A request that composes no document: the table places every row at its
    own index (L_tot = 0), the question is prefilled over itself alone and
    the answer decoded after it."""
    g = S.Geometry(1, 8, 2, 128, 5.0e5)
    Q, T = 20, 3
    sc = Scenario(g, 4, [(1, 40, 10)], [([], None)], q_len=Q, decode_steps=T)
    bt = sc.batch
    assert bt.n_slots == [0] and bt.l_tot == [0]
    bt.compose()
    rng = np.random.default_rng(31)
    q = S.normal_bf16(rng, (1, Q, 8, 128))
    kq = S.normal_bf16(rng, (1, Q, 2, 128))
    vq = S.normal_bf16(rng, (1, Q, 2, 128))
    qd = S.normal_bf16(rng, (T, 1, 8, 128))
    kd = S.normal_bf16(rng, (T, 1, 2, 128))
    vd = S.normal_bf16(rng, (T, 1, 2, 128))
    pre = torch.empty((1, Q, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt.prefill(0, to_dev(q), to_dev(kq), to_dev(vq), pre)
    bt.reset_decode()
    dec = []
    for t in range(T):
        o = torch.empty((1, 8, 128), dtype=torch.bfloat16, device="cuda")
        bt.decode(0, to_dev(qd[t]), to_dev(kd[t]), to_dev(vd[t]), o)
        bt.advance()
        dec.append(o)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    assert np.array_equal(bt.pos[0].cpu().numpy(), np.arange(bt.cap))
    empty = np.zeros((2, 0, 128), np.uint16)
    ref_pre, krot = O.attend_new_tokens(q[0], kq[0], vq[0], empty, empty, 0, g.rope_theta)
    check_attention(pre[0], ref_pre, "question-only prefill")
    check_keys(to_bits(bt.k_caches[0][0, :, :Q]), krot, "question keys")
    ref_dec, kc, vc = O.decode_sequence(qd[:, 0], kd[:, 0], vd[:, 0], krot, vq[0].transpose(1, 0, 2), Q,
                                        g.rope_theta)
    check_attention(torch.stack(dec)[:, 0], ref_dec, "decode after a question-only prefill")
    assert np.array_equal(to_bits(bt.v_caches[0][0, :, :Q + T]), vc)
    sc.close()


def test_compose_orders_repeats_and_ragged_docs():
    """Partial last blocks, a one-slot document, repeated ids, permutations,
    cap equal to N (no tail), rows past N untouched."""
    g = S.Geometry(2, 8, 2, 128, 5.0e5)
    specs = [(7, 3, 1), (8, 10, 3), (9, 401, 101), (10, 64, 16), (11, 33, 9)]
    requests = [([9, 7, 8, 9], [3, 1, 0, 2]), ([10, 11, 7], None), ([8], None)]
    sc = Scenario(g, 4, specs, requests, q_len=0, decode_steps=0)
    bt = sc.batch
    for b in range(len(requests)):
        bt.k_caches[b].fill_(7.0)
        bt.v_caches[b].fill_(7.0)
    bt.compose()
    torch.cuda.synchronize()
    st = sc.oracle_store()
    for b, (ids, order) in enumerate(requests):
        N = bt.n_slots[b]
        _, _, kref, vref = O.compose(st, ids, order, 4, g.rope_theta)
        pos_ref, lt = O.composed_positions([sc.docs[d].n_tokens for d in O.composed_order(ids, order)],
                                           [sc.docs[d].n_slots for d in O.composed_order(ids, order)], 4)
        assert np.array_equal(bt.pos[b][:N].cpu().numpy(), pos_ref)
        assert np.array_equal(to_bits(bt.v_caches[b][:, :, :N]), vref)
        check_keys(to_bits(bt.k_caches[b][:, :, :N]), kref, f"request {b}")
        assert torch.all(bt.k_caches[b][:, :, N:] == 7.0) and torch.all(bt.v_caches[b][:, :, N:] == 7.0)
    # cap exactly N: a direct compose into a tight buffer
    N = bt.n_slots[0]
    kt = torch.empty((2, 2, N, 128), dtype=torch.bfloat16, device="cuda")
    vt = torch.empty_like(kt)
    tab = torch.empty(P.c2kv_rope_table_bytes(g, N) // 4, dtype=torch.float32, device="cuda")
    n, nxt = P.c2kv_compose(sc.store, *requests[0], 4, kt, vt, N, tab)
    torch.cuda.synchronize()
    assert n == N
    assert torch.equal(kt, bt.k_caches[0][:, :, :N]) and torch.equal(vt, bt.v_caches[0][:, :, :N])
    sc.close()


def test_compose_many_tiny_documents():
    """500 documents of 1..9 tokens (1..3 slots at k=4) in a shuffled order, so
    that the composition kernel's 8-slot tiles span several documents each and
    its document lookup runs over a long segment table; the head_dim 64
    instantiation as well as 128."""
    for d in (128, 64):
        g = S.Geometry(2, 8, 2, d, 1.0e4)
        rng = np.random.default_rng(0xC0 + d)
        specs = []
        for i in range(500):
            n = int(rng.integers(1, 10))
            specs.append((i, n, -(-n // 4)))
        order = [int(x) for x in rng.permutation(500)]
        requests = [(list(range(500)), order), (list(range(0, 500, 7)), None)]
        sc = Scenario(g, 4, specs, requests, q_len=0, decode_steps=0)
        bt = sc.batch
        bt.compose()
        torch.cuda.synchronize()
        st = sc.oracle_store()
        for b, (ids, order_b) in enumerate(requests):
            N = bt.n_slots[b]
            _, _, kref, vref = O.compose(st, ids, order_b, 4, g.rope_theta)
            seq = O.composed_order(ids, order_b)
            pos_ref, _ = O.composed_positions([sc.docs[x].n_tokens for x in seq], [sc.docs[x].n_slots for x in seq], 4)
            assert np.array_equal(bt.pos[b][:N].cpu().numpy(), pos_ref)
            assert np.array_equal(to_bits(bt.v_caches[b][:, :, :N]), vref), f"V, request {b}, d {d}"
            check_keys(to_bits(bt.k_caches[b][:, :, :N]), kref, f"request {b}, d {d}")
        sc.close()


def test_k1_composition_equals_uncompressed():
    """k=1 keeps every token: the composed cache and the attention over it must
    equal the plain RoPE cache of the concatenated documents."""
    g = S.Geometry(1, 8, 2, 128, 5.0e5)
    lens = [300, 17, 512, 45]
    sc = Scenario(g, 1, [(i, n, n) for i, n in enumerate(lens)], [([0, 1, 2, 3], [2, 0, 3, 1])],
                  q_len=8, decode_steps=3)
    w = S.Workload("k1", g, 1, 1, 8, 3, doc_tokens=tuple(lens))
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    bt = sc.batch
    assert bt.pos[0][:sum(lens)].cpu().numpy().tolist() == list(range(sum(lens)))
    check_request(sc, inputs, pre, dec, 0, layers=[0], steps=range(3))
    sc.close()


def test_k1_uncompressed_128k_tokens():
    """The 128k-token request uncompressed: 32 documents x 4096 tokens at k=1
    (131 072 slots, one layer).  The position table is 0..131071, and the
    composed cache, a 16-token question and two decode steps over 131 088+
    keys match the oracle: attention over the plain RoPE cache of the
    concatenated documents."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    n = 4096
    specs = [(i, n, n) for i in range(32)]
    sc = Scenario(g, 1, specs, [(list(range(32)), None)], q_len=16, decode_steps=2, seed=0xC2C4)
    w = S.Workload("k1_128k", g, 1, 1, 16, 2, seed=0xC2C4)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    assert sc.batch.n_slots[0] == 32 * n
    assert np.array_equal(sc.batch.pos[0][:32 * n].cpu().numpy(), np.arange(32 * n))
    check_request(sc, inputs, pre, dec, 0, layers=[0], steps=[0, 1])
    sc.close()


def test_varlen_batch_pool():
    """Batch of 16 requests drawn from a document pool in random order
    (lengths 500..4000 tokens, one not a multiple of k) through the full
    32-layer Llama stack (the pool workload's launch configuration: per
    sequence decode splits over 16 composed lengths of ~18 000 slots);
    checked on the first and last layer of three requests."""
    g = S.LLAMA31_8B
    rng = np.random.default_rng(0xC2C2)
    lens = [int(x) for x in rng.choice(np.arange(500, 4001, 4), 40)]
    lens[5] = 1003
    specs = [(i, n, -(-n // 4)) for i, n in enumerate(lens)]
    requests = []
    for _ in range(16):
        ids = [int(x) for x in rng.choice(40, 8, replace=False)]
        requests.append((ids, [int(x) for x in rng.permutation(8)]))
    sc = Scenario(g, 4, specs, requests, q_len=32, decode_steps=4)
    w = S.Workload("pool", g, 4, 16, 32, 4, seed=0xC2C2)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    for b in (0, 5, 15):
        check_request(sc, inputs, pre, dec, b, layers=[0, 31], steps=[0, 3])
    sc.close()


def test_decode_four_128k_token_requests():
    """The largest workload's decode launch: 4 requests of 32 x 4096-token
    documents at k=4 (32 768 slots each, each request in its own order), so
    the key tiles of 4 sequences x 8 kv heads are split over the CTAs and
    merged across CTAs as in the benchmark; every request against the oracle
    on one layer, two decode steps."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    specs = [(i, 4096, 1024) for i in range(32)]
    rng = np.random.default_rng(0xC2C6)
    requests = [(list(range(32)), [int(x) for x in rng.permutation(32)]) for _ in range(4)]
    sc = Scenario(g, 4, specs, requests, q_len=0, decode_steps=2, seed=0xC2C6)
    w = S.Workload("long_b4", g, 4, 4, 0, 2, seed=0xC2C6)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    for b in range(4):
        check_request(sc, inputs, pre, dec, b, layers=[0], steps=[0, 1])
    sc.close()


@pytest.mark.parametrize("batch", [4, 5])
def test_decode_cluster_merge_batches(batch):
    """Batches of 4 and 5 sequences (Llama heads): 32 and 40 (sequence, kv
    head) units leave 4 and 3 key splits per unit, which merge inside a
    thread-block cluster through distributed shared memory."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    rng = np.random.default_rng(40 + batch)
    specs = [(i, int(n), -(-int(n) // 4)) for i, n in enumerate(rng.integers(1500, 4000, 10))]
    requests = [([int(x) for x in rng.choice(10, 3, replace=False)], None) for _ in range(batch)]
    sc = Scenario(g, 4, specs, requests, q_len=16, decode_steps=3)
    w = S.Workload("clusters", g, 4, batch, 16, 3, seed=0xC2C6 + batch)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    for b in range(batch):
        check_request(sc, inputs, pre, dec, b, layers=[0], steps=[0, 2])
    sc.close()


@pytest.mark.parametrize("batch", [1, 4])
def test_decode_wait_timeout_is_reported_and_context_recovers(batch):
    """Failure detection without a fault: the test hook makes a decode launch
    wait ~0.5 ms on a barrier nothing arrives on.  The kernel takes its
    timeout path (global last-CTA merge at batch 1, cluster merge at batch 4),
    the host reads C2KV_ETIMEOUT, and the same step decoded again right after
    matches the oracle."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    specs = [(i, 3000 + 400 * i, 750 + 100 * i) for i in range(4)]
    requests = [([i % 4, (i + 1) % 4], None) for i in range(batch)]
    sc = Scenario(g, 4, specs, requests, q_len=8, decode_steps=1)
    w = S.Workload("timeout", g, 4, batch, 8, 1, seed=0xC2C9 + batch)
    inputs = S.make_step_inputs(w)
    dev = upload(inputs)
    bt = sc.batch
    bt.compose()
    pre = []
    for l in range(g.n_layers):
        o = torch.empty_like(dev["q_pre"][l])
        bt.prefill(l, dev["q_pre"][l], dev["kq_pre"][l], dev["vq"][l], o)
        pre.append(o)
    bt.reset_decode()
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    junk = torch.empty_like(dev["qd_pre"][0, 0])
    P.c2kv_test_expire_next_waits(1)
    bt.decode(0, dev["qd_pre"][0, 0], dev["kd_pre"][0, 0], dev["vd"][0, 0], junk)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_ETIMEOUT
    out = torch.empty_like(junk)
    bt.decode(0, dev["qd_pre"][0, 0], dev["kd_pre"][0, 0], dev["vd"][0, 0], out)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    for b in range(batch):
        check_request(sc, inputs, pre, [[out]], b, layers=[0], steps=[0])
    P.c2kv_test_expire_next_waits(0)
    sc.close()


def test_qwen_group5_k16():
    """Qwen3-14B attention geometry (G=5, theta 1e6) at k=16: 16 x 8000-token
    documents -> 8000 slots, 2 layers, batch 2, 128-token question."""
    g = S.Geometry(2, 40, 8, 128, 1.0e6)
    specs = [(i, 8000, 500) for i in range(16)]
    rng = np.random.default_rng(4)
    requests = [(list(range(16)), None), (list(range(16)), [int(x) for x in rng.permutation(16)])]
    sc = Scenario(g, 16, specs, requests, q_len=128, decode_steps=2)
    w = S.Workload("qwen", g, 16, 2, 128, 2, seed=0xC2C4)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    check_request(sc, inputs, pre, dec, 1, layers=[0], steps=[0, 1])
    sc.close()


def test_qwen_batch8_full_size():
    """The Qwen3-14B workload's launches at full size on one layer: 8
    requests of 16 x 8000-token documents at k=16 (8000 slots each, own
    orders), a 128-token question (320 prefill units: two launches) and two
    decode steps (64 units split over the CTAs); four requests against the
    oracle."""
    g = S.Geometry(1, 40, 8, 128, 1.0e6)
    specs = [(i, 8000, 500) for i in range(16)]
    rng = np.random.default_rng(0xC2C7)
    requests = [(list(range(16)), [int(x) for x in rng.permutation(16)]) for _ in range(8)]
    sc = Scenario(g, 16, specs, requests, q_len=128, decode_steps=2, seed=0xC2C7)
    w = S.Workload("qwen_b8", g, 16, 8, 128, 2, seed=0xC2C7)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    for b in (0, 3, 6, 7):
        check_request(sc, inputs, pre, dec, b, layers=[0], steps=[0, 1])
    sc.close()


def test_llama_8x4000_full_size():
    """The benchmark workload at full size (32 layers, 8000 slots, 64-token
    question, 128 decode steps), checked on sampled layers and steps."""
    w = S.WORKLOADS["llama8b_8x4000_k4"]
    docs, reqs = S.make_requests(w)
    sc = Scenario(w.geom, w.k, [(i, n, s) for i, (n, s) in docs.items()],
                  [(r.doc_ids, r.order) for r in reqs], w.q_len, w.decode_steps, seed=w.seed)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    bt = sc.batch
    N = bt.n_slots[0]
    assert N == 8000 and bt.l_tot[0] == 32000
    # V rows of every layer are the stored segments back to back
    seq = O.composed_order(sc.reqs[0].doc_ids, sc.reqs[0].order)
    vcat = np.concatenate([sc.docs[d].v for d in seq], axis=2)
    assert np.array_equal(to_bits(bt.v_caches[0][:, :, :N]), vcat)
    check_request(sc, inputs, pre, dec, 0, layers=[0, 31], steps=[0, 1, 127])
    sc.close()


def test_llama_8x4000_full_size_sharp_needles():
    """The benchmark workload at full size with a sharp softmax: q scaled by 4
    (so a handful of keys dominate every row instead of a near-uniform spread
    over 8000 keys) and, in every layer and kv head, 16 planted "needle" keys
    pointing along the first decode token's q (of the group's first head)
    once both are rotated to their positions, so at decode step 0 the needles
    take almost all of the weight.  Checked on layers 0 and 31, decode steps 0,
    1 and 127 and every question row, at the same tolerances as the flat case."""
    w = S.WORKLOADS["llama8b_8x4000_k4"]
    g = w.geom
    docs, reqs = S.make_requests(w)
    inputs = S.make_step_inputs(w, q_scale=4.0)
    req = reqs[0]
    seq = O.composed_order(req.doc_ids, req.order)
    pos, l_tot = O.composed_positions([docs[d][0] for d in seq], [docs[d][1] for d in seq], w.k)
    target = l_tot + w.q_len                      # position of decode step 0
    starts = np.cumsum([0] + [docs[d][1] for d in seq])
    needles = np.linspace(5, len(pos) - 9, 16).astype(np.int64)   # composed slot indices
    G = g.n_q_heads // g.n_kv_heads

    def plant(dd):
        for i in needles:
            c = int(np.searchsorted(starts, i, side="right") - 1)
            doc, j = dd[seq[c]], int(i - starts[c])
            # pre-RoPE key k = R(target - pos_i) q0, so that R(pos_i) k = R(target) q0
            q0 = O.bf16_to_f64(inputs.qd_pre[0, :, 0, ::G])           # [L][Hkv][d]
            k = O.rope_rotate(q0, np.array([target - pos[i]] * g.n_kv_heads), g.rope_theta)
            k *= 6.0 / np.linalg.norm(k, axis=-1, keepdims=True)
            doc.k_pre[:, :, j, :] = O.f64_to_bf16(k)

    sc = Scenario(g, w.k, [(i, n, s) for i, (n, s) in docs.items()], [(r.doc_ids, r.order) for r in reqs],
                  w.q_len, w.decode_steps, seed=w.seed, mutate=plant)
    # the planted keys do dominate step 0 (layer 0, head 0): each needle's
    # score exceeds every other composed key's by more than 5 (natural log)
    _, _, k0, _ = O.compose(sc.oracle_store(), req.doc_ids, req.order, w.k, g.rope_theta, layers=[0])
    qr = O.rope_rotate(O.bf16_to_f64(inputs.qd_pre[0, 0, 0, :1]), np.array([target]), g.rope_theta)[0]
    sc0 = O.bf16_to_f64(k0[0, 0]) @ qr / np.sqrt(g.head_dim)
    others = np.delete(sc0, needles)
    assert sc0[needles].min() - others.max() > 5.0, (sc0[needles].min(), others.max())
    pre, dec = run_all(sc, upload(inputs))
    check_request(sc, inputs, pre, dec, 0, layers=[0, 31], steps=[0, 1, 127])
    sc.close()


def test_decode_multi_split_long_cache():
    """One long sequence (32768 slots as in the 128k-token workload, 1 layer):
    many key splits merged by the last-arriving CTA."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    specs = [(i, 4096, 1024) for i in range(32)]
    sc = Scenario(g, 4, specs, [(list(range(32)), None)], q_len=0, decode_steps=3)
    w = S.Workload("long", g, 4, 1, 0, 3, seed=0xC2C3)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    check_request(sc, inputs, pre, dec, 0, layers=[0], steps=[0, 2])
    sc.close()


@pytest.mark.parametrize("n_doc,n_slot,k", [(12, 3, 4), (200, 50, 4), (257, 17, 16), (40, 40, 1), (1, 0, 4)])
def test_structured_mask_mode(n_doc, n_slot, k):
    g = S.TINY
    rng = np.random.default_rng(n_doc * 131 + n_slot)
    N = n_doc + n_slot
    q = S.normal_bf16(rng, (N, g.n_q_heads, g.head_dim))
    kk = S.normal_bf16(rng, (N, g.n_kv_heads, g.head_dim))
    v = S.normal_bf16(rng, (N, g.n_kv_heads, g.head_dim))
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, g.n_q_heads, g.head_dim), dtype=torch.bfloat16, device="cuda")
    P.c2kv_attend_masked(g, P.C2KV_MASK_STRUCTURED, n_doc, n_slot, k, to_dev(q), to_dev(kk), to_dev(v), out, ws)
    torch.cuda.synchronize()
    ref = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, g.rope_theta)
    check_attention(out, ref, f"structured mask {n_doc}+{n_slot} k={k}")


def test_structured_mask_extraction_full_size():
    """A 4000-token document with its 1000 slots (k=4) under the structured
    mask, Llama3.1-8B heads: slot tiles skip the document key tiles they
    cannot see.  The oracle computes sampled rows: document rows, slot rows at
    tile edges, the last slot and random ones."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    n_doc, k = 4000, 4
    n_slot = O.slot_count(n_doc, k)
    N = n_doc + n_slot
    rng = np.random.default_rng(17)
    q = S.normal_bf16(rng, (N, 32, 128))
    kk = S.normal_bf16(rng, (N, 8, 128))
    v = S.normal_bf16(rng, (N, 8, 128))
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, 32, 128), dtype=torch.bfloat16, device="cuda")
    P.c2kv_attend_masked(g, P.C2KV_MASK_STRUCTURED, n_doc, n_slot, k, to_dev(q), to_dev(kk), to_dev(v), out, ws)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    rows = [0, 1, 63, 64, 1000, 3999, 4000, 4001, 4031, 4032, 4063, 4064, 4500, N - 1]
    rows += sorted(rng.choice(N, 18, replace=False).tolist())
    ref = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, g.rope_theta, rows=rows)
    check_attention(out[rows], ref, "structured mask 4000 + 1000, k=4")


@pytest.mark.parametrize("n_doc,n_slot,k", [(12, 3, 4), (200, 50, 4), (257, 17, 16), (40, 40, 1),
                                             (600, 150, 4), (300, 0, 4), (1, 0, 4)])
def test_anchor_mask_mode(n_doc, n_slot, k):
    """The anchor-token ablation: document rows see their causal prefix and
    every anchor (the key tiles in between are skipped), anchors see the
    document and earlier anchors.  (600, 150) leaves dead key tiles between
    the first document rows and the anchors; n_slot = 0 is plain causal
    attention, and a single token takes the one-token path."""
    g = S.TINY
    rng = np.random.default_rng(n_doc * 137 + n_slot)
    N = n_doc + n_slot
    q = S.normal_bf16(rng, (N, g.n_q_heads, g.head_dim))
    kk = S.normal_bf16(rng, (N, g.n_kv_heads, g.head_dim))
    v = S.normal_bf16(rng, (N, g.n_kv_heads, g.head_dim))
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, g.n_q_heads, g.head_dim), dtype=torch.bfloat16, device="cuda")
    P.c2kv_attend_masked(g, P.C2KV_MASK_ANCHOR, n_doc, n_slot, k, to_dev(q), to_dev(kk), to_dev(v), out, ws)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    ref = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, g.rope_theta, mask="anchor")
    check_attention(out, ref, f"anchor mask {n_doc}+{n_slot} k={k}")


@pytest.mark.parametrize("mask", ["structured", "anchor"])
@pytest.mark.parametrize("hq,hkv,d", [(40, 8, 128), (8, 8, 128), (16, 2, 64)])
def test_masked_modes_group_sizes(hq, hkv, d, mask):
    """Both extraction masks at G = 5 (25 tokens per 125-row M tile), G = 1
    and G = 8, with the document/slot boundary inside an M tile."""
    g = S.Geometry(1, hq, hkv, d, 1.0e6)
    n_doc, k = 310, 4
    n_slot = O.slot_count(n_doc, k)
    N = n_doc + n_slot
    rng = np.random.default_rng(hq * 7 + hkv + d)
    q = S.normal_bf16(rng, (N, hq, d))
    kk = S.normal_bf16(rng, (N, hkv, d))
    v = S.normal_bf16(rng, (N, hkv, d))
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, hq, d), dtype=torch.bfloat16, device="cuda")
    code = P.C2KV_MASK_STRUCTURED if mask == "structured" else P.C2KV_MASK_ANCHOR
    P.c2kv_attend_masked(g, code, n_doc, n_slot, k, to_dev(q), to_dev(kk), to_dev(v), out, ws)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    ref = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, g.rope_theta, mask=mask)
    check_attention(out, ref, f"{mask} mask, {hq}/{hkv} heads, d={d}")


def test_anchor_mask_extraction_full_size():
    """A 4000-token document with 1000 anchor tokens (k=4 positions) under the
    anchor-token mask, Llama3.1-8B heads, sampled rows: early document rows
    (most key tiles dead), rows at M-tile edges, the last document row, the
    first and last anchors and random ones."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    n_doc, k = 4000, 4
    n_slot = O.slot_count(n_doc, k)
    N = n_doc + n_slot
    rng = np.random.default_rng(23)
    q = S.normal_bf16(rng, (N, 32, 128))
    kk = S.normal_bf16(rng, (N, 8, 128))
    v = S.normal_bf16(rng, (N, 8, 128))
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, 32, 128), dtype=torch.bfloat16, device="cuda")
    P.c2kv_attend_masked(g, P.C2KV_MASK_ANCHOR, n_doc, n_slot, k, to_dev(q), to_dev(kk), to_dev(v), out, ws)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    rows = [0, 1, 15, 16, 127, 128, 2047, 3968, 3999, 4000, 4001, 4015, 4016, N - 1]
    rows += sorted(rng.choice(N, 18, replace=False).tolist())
    ref = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, g.rope_theta, rows=rows, mask="anchor")
    check_attention(out[rows], ref, "anchor mask 4000 + 1000, k=4")


def test_causal_mask_mode_llama_heads():
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    N = 300
    rng = np.random.default_rng(3)
    q = S.normal_bf16(rng, (N, 32, 128))
    kk = S.normal_bf16(rng, (N, 8, 128))
    v = S.normal_bf16(rng, (N, 8, 128))
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, 32, 128), dtype=torch.bfloat16, device="cuda")
    P.c2kv_attend_masked(g, P.C2KV_MASK_CAUSAL, N, 0, 1, to_dev(q), to_dev(kk), to_dev(v), out, ws)
    torch.cuda.synchronize()
    ref = O.masked_extraction_attention(q, kk, v, N, 0, 1, g.rope_theta)
    check_attention(out, ref, "causal mask mode")


def test_continue_tracks_the_most_recent_tables():
    """The store remembers the compositions into the 1024 tables composed into
    most recently: after 1025 compositions into distinct tables, continuing
    the first one is refused and continuing the second and the last works."""
    g = S.Geometry(2, 4, 2, 64, 1.0e4)
    k = 4
    doc = S.make_document(g, 1, 8, k, 3)
    store = P.c2kv_store_create(g, 1 << 20)
    try:
        P.c2kv_store_segments(store, [1], [doc.n_tokens], [doc.n_slots], k, [doc.k_pre], [doc.v])
        cap = doc.n_slots
        kc = torch.zeros((g.n_layers, g.n_kv_heads, cap, g.head_dim), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        tb = P.c2kv_rope_table_bytes(g, cap)
        n = 1025
        tabs = torch.zeros((n, tb), dtype=torch.uint8, device="cuda")
        for i in range(n):
            P.c2kv_compose_layers(store, [1], None, k, 0, 0, 1, kc, vc, cap, tabs[i])
        with pytest.raises(P.C2KVError) as e:
            P.c2kv_compose_layers(store, [1], None, k, P.C2KV_COMPOSE_CONTINUE, 1, 2, kc, vc, cap, tabs[0])
        assert e.value.status == P.C2KV_EINVAL
        for i in (1, n - 1):
            P.c2kv_compose_layers(store, [1], None, k, P.C2KV_COMPOSE_CONTINUE, 1, 2, kc, vc, cap, tabs[i])
        torch.cuda.synchronize()
        assert P.c2kv_device_error() == P.C2KV_OK
    finally:
        P.c2kv_store_destroy(store)


def test_store_save_and_load_round_trip(tmp_path):
    """A saved store, loaded into a new one, composes the same caches bit for
    bit; documents stored at different k keep theirs.  Files of another
    geometry, truncated files, missing files and ids already stored are
    rejected."""
    g = S.Geometry(2, 8, 2, 128, 5.0e5)
    docs4 = {i: S.make_document(g, i, n, 4, 0xC2CA) for i, n in ((1, 401), (2, 64), (3, 1000))}
    docs16 = {7: S.make_document(g, 7, 320, 16, 0xC2CA)}
    pool = sum(2 * d.k_pre.nbytes + 1024 for d in list(docs4.values()) + list(docs16.values())) + (1 << 20)
    a = P.c2kv_store_create(g, pool)
    for k, docs in ((4, docs4), (16, docs16)):
        ids = list(docs)
        P.c2kv_store_segments(a, ids, [docs[i].n_tokens for i in ids], [docs[i].n_slots for i in ids], k,
                              [docs[i].k_pre for i in ids], [docs[i].v for i in ids])
    path = str(tmp_path / "store.c2kv")
    P.c2kv_store_save(a, path)
    b = P.c2kv_store_create(g, pool)
    P.c2kv_store_load(b, path)
    for i in (1, 2, 3, 7):
        assert P.c2kv_store_lookup(a, i) == P.c2kv_store_lookup(b, i)
    caches = []
    for st in (a, b):
        kc = torch.full((2, 2, 2048, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        vc = torch.full_like(kc, 7.0)
        tab = torch.empty(P.c2kv_rope_table_bytes(g, 2048) // 4, dtype=torch.float32, device="cuda")
        P.c2kv_compose(st, [3, 1, 2, 1], [1, 0, 3, 2], 4, kc, vc, 2048, tab)
        caches.append((kc, vc))
    torch.cuda.synchronize()
    assert torch.equal(caches[0][0], caches[1][0]) and torch.equal(caches[0][1], caches[1][1])
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_store_load(b, path)                        # ids already stored
    assert e.value.status == P.C2KV_EINVAL
    other = P.c2kv_store_create(S.Geometry(2, 8, 2, 64, 5.0e5), 1 << 20)
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_store_load(other, path)
    assert e.value.status == P.C2KV_EINVAL
    raw = open(path, "rb").read()
    cut = str(tmp_path / "cut.c2kv")
    open(cut, "wb").write(raw[:len(raw) // 2])
    c = P.c2kv_store_create(g, pool)
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_store_load(c, cut)
    assert e.value.status == P.C2KV_EIO
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_store_load(c, str(tmp_path / "missing.c2kv"))
    assert e.value.status == P.C2KV_EIO
    for st in (a, b, c, other):
        P.c2kv_store_destroy(st)


def test_host_side_errors():
    g = S.Geometry(1, 8, 2, 128, 5.0e5)
    sc = Scenario(g, 4, [(1, 40, 10), (2, 8, 2)], [([1, 2], None)], q_len=4, decode_steps=2)
    kc = torch.empty((1, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    tab = torch.empty(P.c2kv_rope_table_bytes(g, 16) // 4, dtype=torch.float32, device="cuda")
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_compose(sc.store, [1, 2], None, 4, kc, vc, 11, tab)
    assert e.value.status == P.C2KV_ECAPACITY
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_compose(sc.store, [1, 99], None, 4, kc, vc, 16, tab)
    assert e.value.status == P.C2KV_ENOTFOUND
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_compose(sc.store, [1, 2], None, 8, kc, vc, 16, tab)
    assert e.value.status == P.C2KV_EINVAL
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_compose(sc.store, [1, 2], [1, 1], 4, kc, vc, 16, tab)
    assert e.value.status == P.C2KV_EINVAL
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_store_segments(sc.store, [1], [40], [10], 4, [sc.docs[1].k_pre], [sc.docs[1].v])
    assert e.value.status == P.C2KV_EINVAL
    bt = sc.batch
    q = torch.zeros((1, 5, 8, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((1, 5, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_attend_prefill(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, [bt.cap - 2], q, kn, kn,
                              torch.empty_like(q), bt.workspace)
    assert e.value.status == P.C2KV_ECAPACITY
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_attend_prefill(g, 1, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, [0], q, kn, kn,
                              torch.empty_like(q), bt.workspace)
    assert e.value.status == P.C2KV_EINVAL
    sc.close()


def test_device_length_beyond_capacity_is_reported():
    """A device-side length past the cache capacity is caught by the kernels:
    the output is skipped and c2kv_device_error reports C2KV_EDEVICE."""
    g = S.Geometry(1, 8, 2, 128, 5.0e5)
    sc = Scenario(g, 4, [(1, 40, 10)], [([1], None)], q_len=0, decode_steps=2)
    bt = sc.batch
    bt.compose()
    bt.reset_decode()
    bt.n_cached_dev.fill_(bt.cap)   # no room for the new token
    q = torch.ones((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.ones((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, 3.0)
    bt.decode(0, q, kn, kn, out)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_EDEVICE
    assert torch.all(out == 3.0)
    assert P.c2kv_device_error() == P.C2KV_OK   # reading clears the word
    sc.close()


def test_prefill_units_beyond_one_wave():
    """A question whose (sequence, M tile, kv head) units outnumber the SMs:
    Qwen3-14B heads (G = 5), 8 requests x 128 tokens = 320 units.  Whole
    waves run unsplit and the rest of the last wave runs as key-split
    clusters in a second launch (on 152 SMs: 304 units, then 16); every
    request's question rows and a decode step against the oracle."""
    g = S.Geometry(1, 40, 8, 128, 1.0e6)
    specs = [(i, 1200 + 48 * i, 300 + 12 * i) for i in range(8)]
    sc = Scenario(g, 4, specs, [([i], None) for i in range(8)], q_len=128, decode_steps=1)
    w = S.Workload("qwen_waves", g, 4, 8, 128, 1, seed=0xC2C5)
    inputs = S.make_step_inputs(w)
    dev = upload(inputs)
    bt = sc.batch
    bt.compose()
    out = torch.empty_like(dev["q_pre"][0])
    n0 = P.c2kv_kernel_launches()
    bt.prefill(0, dev["q_pre"][0], dev["kq_pre"][0], dev["vq"][0], out)
    launches = P.c2kv_kernel_launches() - n0
    bt.reset_decode()
    dec = torch.empty_like(dev["qd_pre"][0, 0])
    bt.decode(0, dev["qd_pre"][0, 0], dev["kd_pre"][0, 0], dev["vd"][0, 0], dec)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert launches == 3, launches   # the question's append, then the two prefill launches
    for b in range(8):
        check_request(sc, inputs, [out], [[dec]], b, layers=[0], steps=[0])
    sc.close()


@pytest.mark.parametrize("hq,hkv,d,q_len", [(8, 8, 128, 40), (16, 2, 128, 33), (4, 2, 64, 1), (8, 1, 64, 130)])
def test_prefill_group_sizes_and_ragged_tiles(hq, hkv, d, q_len):
    """Tensor-core prefill for G = 1 and 8, a ragged last M tile, a one-token
    question (which takes the CUDA-core path) and a single kv head."""
    g = S.Geometry(1, hq, hkv, d, 1.0e4)
    specs = [(1, 700, 175), (2, 13, 4)]
    sc = Scenario(g, 4, specs, [([2, 1], None)], q_len=q_len, decode_steps=2)
    w = S.Workload("g", g, 4, 1, q_len, 2, seed=hq * 100 + q_len)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    check_request(sc, inputs, pre, dec, 0, layers=[0], steps=[0, 1])
    sc.close()


def test_rope_table_matches_fp64_angles():
    """The per-row cos/sin table (hi + lo fp32 pairs) against the oracle's fp64
    cos/sin of pos * theta^(-2i/d), at positions up to ~1.3e5."""
    for g in (S.Geometry(1, 32, 8, 128, 5.0e5), S.Geometry(1, 4, 2, 64, 1.0e4)):
        pos = np.array([0, 1, 3, 7, 403, 32000, 99991, 131071, 131072 + 255], dtype=np.int32)
        tab = torch.empty(P.c2kv_rope_table_bytes(g, len(pos)) // 4, dtype=torch.float32, device="cuda")
        P.c2kv_rope_table(g, torch.from_numpy(pos).cuda(), tab)
        torch.cuda.synchronize()
        t = tab.cpu().numpy().astype(np.float64).reshape(len(pos), g.head_dim // 2, 4)
        ang = pos.astype(np.float64)[:, None] * O.rope_inv_freq(g.rope_theta, g.head_dim)[None, :]
        assert np.abs(t[..., 0] + t[..., 1] - np.cos(ang)).max() < 1e-12
        assert np.abs(t[..., 2] + t[..., 3] - np.sin(ang)).max() < 1e-12
        # the hi parts alone are the fp32-rounded values
        assert np.abs(t[..., 0] - np.cos(ang)).max() < 1e-7


def test_decode_overlapped_launches_match_serial_ones():
    """Layer > 0 decode launches may start while the previous layer's decode
    finishes (C2KV_DECODE_OVERLAP_PREVIOUS); the results must be identical to
    fully serialised launches."""
    g = S.Geometry(4, 32, 8, 128, 5.0e5)
    specs = [(i, 4000, 1000) for i in range(4)]
    w = S.Workload("ovl", g, 4, 1, 0, 3, seed=0xC2C5)
    inputs = upload(S.make_step_inputs(w))
    outs = []
    for overlap in (False, True):
        sc = Scenario(g, 4, specs, [(list(range(4)), [2, 0, 3, 1])], q_len=0, decode_steps=3, seed=0xC2C5)
        bt = sc.batch
        bt.compose()
        bt.reset_decode()
        res = []
        for t in range(3):
            for l in range(4):
                o = torch.empty_like(inputs["qd_pre"][t, l])
                bt.decode(l, inputs["qd_pre"][t, l], inputs["kd_pre"][t, l], inputs["vd"][t, l], o,
                          overlap_previous=overlap and l > 0)
                res.append(o)
            bt.advance()
        torch.cuda.synchronize()
        assert P.c2kv_device_error() == P.C2KV_OK
        outs.append(torch.stack(res).cpu())
        sc.close()
    assert torch.equal(outs[0], outs[1])
