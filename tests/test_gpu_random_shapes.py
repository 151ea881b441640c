"""Seeded random shapes through the whole path (compose, question prefill,
decode) against the oracle: group sizes 1/2/4/5/8, head_dim 64 and 128,
k from 1 to 16, ragged documents, repeated and reordered documents,
requests without documents, one-token and long questions, batches up to 12.
Each case is small, so the planner's corners (one split, cluster splits,
several waves, a key range shorter than a tile) come from the mix rather
than from size.  Same bars as the parity tests."""
import numpy as np
import pytest

from compressed_composable_kv_gb300 import synth as S
from gpu_util import Scenario, check_request, run_all, upload

pytestmark = pytest.mark.gpu


def _case(i: int):
    rng = np.random.default_rng(0xC2C8 + i)
    G = int(rng.choice([1, 2, 4, 5, 8]))
    n_kv = int(rng.choice([1, 2, 4, 8]))
    d = int(rng.choice([64, 128]))
    theta = float(rng.choice([1.0e4, 5.0e5, 1.0e6]))
    layers = int(rng.choice([1, 2]))
    g = S.Geometry(layers, G * n_kv, n_kv, d, theta)
    k = int(rng.choice([1, 2, 4, 8, 16]))
    n_docs = int(rng.integers(1, 7))
    lens = [int(rng.integers(1, 1500)) for _ in range(n_docs)]
    specs = [(j, n, -(-n // k)) for j, n in enumerate(lens)]
    batch = int(rng.integers(1, 13))
    requests = []
    for _ in range(batch):
        m = int(rng.integers(0, n_docs + 2))
        ids = [int(x) for x in rng.integers(0, n_docs, m)]   # repeats allowed, may be empty
        order = [int(x) for x in rng.permutation(m)] if m > 1 and rng.random() < 0.5 else None
        requests.append((ids, order))
    q_len = int(rng.choice([0, 1, int(rng.integers(2, 64)), int(rng.integers(64, 300))]))
    steps = int(rng.integers(1, 4))
    return g, k, specs, requests, q_len, steps, 0xC2C8 + i


CASES = [_case(i) for i in range(48)]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_random_shape(i):
    g, k, specs, requests, q_len, steps, seed = CASES[i]
    sc = Scenario(g, k, specs, requests, q_len=q_len, decode_steps=steps, seed=seed)
    w = S.Workload(f"random{i}", g, k, len(requests), q_len, steps, seed=seed)
    inputs = S.make_step_inputs(w)
    pre, dec = run_all(sc, upload(inputs))
    B = len(requests)
    for b in sorted({0, B // 2, B - 1}):
        check_request(sc, inputs, pre, dec, b, layers=[g.n_layers - 1], steps=range(steps))
    sc.close()
