"""Shared helpers of the GPU parity tests: seeded inputs go to both the CUDA
path (through the C ABI) and the CPU oracle; results are compared here."""
import numpy as np
import torch

import oracle.c2kv_oracle as O
import compressed_composable_kv_gb300 as P
from compressed_composable_kv_gb300 import synth as S

# Tolerances on bf16 attention outputs (fp32 accumulation) against the fp64
# oracle, and on re-rotated keys.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
MAX_ULP = 1


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_attention(gpu_bf16: torch.Tensor, ref: np.ndarray, what: str, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = O.bf16_to_f64(to_bits(gpu_bf16)).reshape(ref.shape)
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref ** 2))) + 1e-30
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.3e}"
    # relative to the output's own scale (near-uniform softmax makes |out| small)
    assert err.mean() / rms <= 2e-2, f"{what}: mean err / rms {err.mean() / rms:.3e}"
    return float(err.max()), float(err.mean())


def check_keys(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str):
    d = O.bf16_ulp_distance(gpu_bits, ref_bits)
    assert d.max() <= MAX_ULP, f"{what}: {int((d > MAX_ULP).sum())} keys off by > {MAX_ULP} ulp (max {d.max()})"


class Scenario:
    """Documents, store and per-request device state of one test workload."""

    def __init__(self, geom, k, doc_specs, requests, q_len, decode_steps, seed=0xC2C0, layers=None,
                 cap_multiple=32, realign=True):
        self.geom, self.k, self.seed, self.realign = geom, k, seed, realign
        self.docs = {}
        for doc_id, n_tok, n_slot in doc_specs:
            self.docs[doc_id] = S.make_document(geom, doc_id, n_tok, k, seed, n_slots=n_slot, layers=layers)
        pool = sum(2 * d.k_pre.nbytes + 1024 for d in self.docs.values()) + (1 << 20)
        self.store = P.c2kv_store_create(geom, pool)
        ids = list(self.docs)
        P.c2kv_store_segments(self.store, ids, [self.docs[i].n_tokens for i in ids],
                              [self.docs[i].n_slots for i in ids], k,
                              [self.docs[i].k_pre for i in ids], [self.docs[i].v for i in ids])
        self.reqs = [P.RequestSpec(list(r[0]), None if r[1] is None else list(r[1])) for r in requests]
        self.batch = P.RequestBatch(self.store, geom, self.reqs, k, q_len, decode_steps,
                                    cap_multiple=cap_multiple, realign=realign)

    def oracle_store(self):
        return {i: (d.n_tokens, d.n_slots, d.k_pre, d.v) for i, d in self.docs.items()}

    def close(self):
        torch.cuda.synchronize()
        P.c2kv_store_destroy(self.store)
