"""The seeded synthetic inputs both sides draw from: deterministic per
document, shaped as the workloads state, and free of the method's
arithmetic (only random numbers and shapes)."""
import numpy as np
import pytest

from compressed_composable_kv_gb300 import synth as S


def test_a_document_has_the_same_bytes_wherever_it_is_drawn():
    g = S.Geometry(2, 4, 2, 64, 1.0e4)
    a = S.make_document(g, 7, 400, 4, 0xC2C0)
    b = S.make_document(g, 7, 400, 4, 0xC2C0)
    c = S.make_document(g, 8, 400, 4, 0xC2C0)
    assert np.array_equal(a.k_pre, b.k_pre) and np.array_equal(a.v, b.v)
    assert not np.array_equal(a.k_pre, c.k_pre)
    assert not np.array_equal(a.k_pre, a.v)
    # one slot per k tokens; a one-layer draw (the oracle's timing sample) keeps the other sizes
    one = S.make_document(g, 7, 400, 4, 0xC2C0, layers=1)
    assert a.k_pre.shape == (2, 2, 100, 64) and one.k_pre.shape == one.v.shape == (1, 2, 100, 64)


def test_values_are_standard_normal_bf16():
    rng = np.random.default_rng(0)
    bits = S.normal_bf16(rng, (200_000,))
    x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.all(np.isfinite(x))


def test_pool_workload_recipe():
    """Batch 16; 8 distinct pool documents per request in a random order;
    lengths multiples of k in [500, 4000]; one slot per k tokens."""
    w = S.WORKLOADS["llama8b_pool256_b16_k4"]
    docs, reqs = S.make_requests(w)
    assert len(docs) == 256 and len(reqs) == 16
    for n, s in docs.values():
        assert 500 <= n <= 4000 and n % w.k == 0 and s == n // w.k
    for r in reqs:
        assert len(r.doc_ids) == 8 and len(set(r.doc_ids)) == 8
        assert sorted(r.order) == list(range(8))
    assert any(r.order != list(range(8)) for r in reqs)
    again, reqs2 = S.make_requests(w)
    assert again == docs and [(r.doc_ids, r.order) for r in reqs2] == [(r.doc_ids, r.order) for r in reqs]


@pytest.mark.parametrize("name,slots", [("tiny", [113]), ("llama8b_8x4000_k4", [8000]),
                                        ("llama8b_32x4096_k4_b4", [32768] * 4),
                                        ("qwen14b_16x8000_k16_b8", [8000] * 8)])
def test_fixed_workloads_compose_the_stated_slot_counts(name, slots):
    w = S.WORKLOADS[name]
    docs, reqs = S.make_requests(w)
    assert [sum(docs[d][1] for d in r.doc_ids) for r in reqs] == slots


def test_step_input_shapes():
    w = S.WORKLOADS["tiny"]
    inp = S.make_step_inputs(w, decode_steps=3)
    g = w.geom
    assert inp.q_pre.shape == (1, 1, 8, g.n_q_heads, g.head_dim)
    assert inp.kq_pre.shape == inp.vq.shape == (1, 1, 8, g.n_kv_heads, g.head_dim)
    assert inp.qd_pre.shape == (3, 1, 1, g.n_q_heads, g.head_dim)
    assert inp.kd_pre.shape == inp.vd.shape == (3, 1, 1, g.n_kv_heads, g.head_dim)
