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
    assert gpu_bits.shape == ref_bits.shape, f"{what}: shapes {gpu_bits.shape} vs {ref_bits.shape}"
    if gpu_bits.size == 0:   # a composition of no documents
        return
    d = O.bf16_ulp_distance(gpu_bits, ref_bits)
    assert d.max() <= MAX_ULP, f"{what}: {int((d > MAX_ULP).sum())} keys off by > {MAX_ULP} ulp (max {d.max()})"


class Scenario:
    """Documents, store and per-request device state of one test workload."""

    def __init__(self, geom, k, doc_specs, requests, q_len, decode_steps, seed=0xC2C0, layers=None,
                 cap_multiple=32, realign=True, mutate=None):
        """mutate(docs): edits the drawn documents before they are stored
        (planted keys); the oracle reads the same edited arrays."""
        self.geom, self.k, self.seed, self.realign = geom, k, seed, realign
        self.docs = {}
        for doc_id, n_tok, n_slot in doc_specs:
            self.docs[doc_id] = S.make_document(geom, doc_id, n_tok, k, seed, n_slots=n_slot, layers=layers)
        if mutate is not None:
            mutate(self.docs)
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


def upload(inputs: S.StepInputs):
    return {name: to_dev(getattr(inputs, name)) for name in
            ("q_pre", "kq_pre", "vq", "qd_pre", "kd_pre", "vd")}


def run_all(sc: Scenario, dev):
    """Compose, prefill every layer, decode every step (the bench's launch
    configuration, without graphs).  Returns the output tensors."""
    bt = sc.batch
    L = sc.geom.n_layers
    bt.compose()
    pre = []
    if bt.q_len:
        for l in range(L):
            out = torch.empty_like(dev["q_pre"][l])
            bt.prefill(l, dev["q_pre"][l], dev["kq_pre"][l], dev["vq"][l], out)
            pre.append(out)
    bt.reset_decode()
    dec = []
    for t in range(bt.decode_steps):
        row = []
        for l in range(L):
            out = torch.empty_like(dev["qd_pre"][t, l])
            bt.decode(l, dev["qd_pre"][t, l], dev["kd_pre"][t, l], dev["vd"][t, l], out)
            row.append(out)
        bt.advance()
        dec.append(row)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    return pre, dec


def check_request(sc: Scenario, inputs: S.StepInputs, pre, dec, b: int, layers, steps):
    bt = sc.batch
    g = sc.geom
    req = sc.reqs[b]
    st = sc.oracle_store()
    N, lt, Q = bt.n_slots[b], bt.l_tot[b], bt.q_len
    seq = O.composed_order(req.doc_ids, req.order)
    pos_ref, lt_ref = O.composed_positions([sc.docs[d].n_tokens for d in seq],
                                           [sc.docs[d].n_slots for d in seq], sc.k, sc.realign)
    assert lt_ref == lt
    assert np.array_equal(bt.pos[b][:N].cpu().numpy(), pos_ref)
    kc = bt.k_caches[b]
    vc = bt.v_caches[b]
    for l in layers:
        _, _, kref, vref = O.compose(st, req.doc_ids, req.order, sc.k, g.rope_theta, layers=[l],
                                     realign=sc.realign)
        kg = to_bits(kc[l, :, :N])
        vg = to_bits(vc[l, :, :N])
        assert np.array_equal(vg, vref[0]), f"V rows differ (layer {l})"
        check_keys(kg, kref[0], f"composed K layer {l}")
        kcache, vcache = kref[0], vref[0]
        if Q:
            o_ref, kq_rot = O.attend_new_tokens(inputs.q_pre[l, b], inputs.kq_pre[l, b], inputs.vq[l, b],
                                                kcache, vcache, lt, g.rope_theta)
            check_attention(pre[l][b], o_ref, f"prefill layer {l} seq {b}")
            check_keys(to_bits(kc[l, :, N:N + Q]), kq_rot, f"question keys layer {l}")
            assert np.array_equal(to_bits(vc[l, :, N:N + Q]), inputs.vq[l, b].transpose(1, 0, 2))
            kcache = np.concatenate([kcache, kq_rot], axis=1)
            vcache = np.concatenate([vcache, inputs.vq[l, b].transpose(1, 0, 2)], axis=1)
        for t in steps:
            if t > 0:
                prev_pos = lt + Q + np.arange(t)
                kd = O.rotate_keys_bf16(inputs.kd_pre[:t, l, b], prev_pos, g.rope_theta)
                kc_t = np.concatenate([kcache, kd], axis=1)
                vc_t = np.concatenate([vcache, inputs.vd[:t, l, b].transpose(1, 0, 2)], axis=1)
            else:
                kc_t, vc_t = kcache, vcache
            o_ref, kn = O.attend_new_tokens(inputs.qd_pre[t:t + 1, l, b], inputs.kd_pre[t:t + 1, l, b],
                                            inputs.vd[t:t + 1, l, b], kc_t, vc_t, lt + Q + t, g.rope_theta)
            check_attention(dec[t][l][b], o_ref[0], f"decode layer {l} step {t} seq {b}")
            row = N + Q + t
            check_keys(to_bits(kc[l, :, row:row + 1]), kn, f"decode key layer {l} step {t}")
