"""The synthetic-weight decoder step (linear layers, RMSNorm, one decoder layer
around the composed-cache attention) through the C ABI against the fp64 CPU
oracle (oracle/decoder_oracle.py).

Bars: a linear layer, an RMSNorm or a SwiGLU output is one bf16 rounding of
an fp32 computation, so it must be within 1 bf16 ulp of the oracle's value
(an fp32 sum can cross a rounding boundary the exact sum does not), or,
where cancellation makes the value tiny, within 2^-14 of the output's RMS.
A whole layer adds the attention's bar (max-abs 2e-2, mean-abs 2e-3 on
outputs of magnitude <= ~1) to the residual stream, plus its bf16 roundings:
max-abs 4e-2 and mean-abs 4e-3 on the layer output.
"""
import numpy as np
import pytest
import torch

import oracle.c2kv_oracle as O
import oracle.decoder_oracle as DO
import compressed_composable_kv_gb300 as P
from compressed_composable_kv_gb300 import synth as S
from gpu_util import Scenario, check_attention, to_bits, to_dev

pytestmark = pytest.mark.gpu


def check_rounded(gpu: torch.Tensor, ref: np.ndarray, what: str):
    got = to_bits(gpu).reshape(ref.shape)
    dist = O.bf16_ulp_distance(got, O.f64_to_bf16(ref))
    err = np.abs(O.bf16_to_f64(got) - ref)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bad = (dist > 1) & (err > 2.0 ** -14 * rms)
    assert not bad.any(), f"{what}: {int(bad.sum())} values off by > 1 ulp (max {err[bad].max():.3e})"
    assert np.all(np.isfinite(O.bf16_to_f64(got))), f"{what}: non-finite"
    return float((dist > 0).mean())


def _ws(tokens, n_out):
    ws = torch.zeros(P.c2kv_linear_workspace_size(tokens, n_out), dtype=torch.uint8, device="cuda")
    P.c2kv_workspace_init(ws)
    return ws


# (tokens, k_in, n_out): a decode batch on the Llama projections; one tile over
# 224 K chunks (152 CTAs' partials merged); 6 chunks over 152 CTAs (most own
# nothing) with 100 tokens (padded to 112); a question of 64 tokens; the
# vocabulary-sized LM head
LINEAR_SHAPES = [(4, 4096, 6144), (1, 4096, 4096), (4, 14336, 128), (100, 128, 384), (64, 4096, 14336 * 2),
                 (4, 4096, 128256)]


@pytest.mark.parametrize("tokens,k_in,n_out", LINEAR_SHAPES)
def test_linear_store_and_add(tokens, k_in, n_out):
    rng = np.random.default_rng(tokens * 7 + n_out)
    x = S.normal_bf16(rng, (tokens, k_in))
    w = S.normal_bf16(rng, (n_out, k_in), k_in ** -0.5)
    r = S.normal_bf16(rng, (tokens, n_out))
    ws = _ws(tokens, n_out)
    xd, wd = to_dev(x), to_dev(w)
    y = torch.empty((tokens, n_out), dtype=torch.bfloat16, device="cuda")
    P.c2kv_linear(xd, wd, y, ws)
    ref = DO.linear(x, w)
    check_rounded(y, ref, f"linear {tokens}x{k_in}x{n_out}")
    # in place: y = x W^T + y
    y2 = to_dev(r)
    P.c2kv_linear(xd, wd, y2, ws, P.C2KV_LINEAR_ADD, residual=y2)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    check_rounded(y2, ref + O.bf16_to_f64(r), f"linear + residual {tokens}x{k_in}x{n_out}")


def test_linear_split3_and_swiglu():
    """The fused QKV projection of the Llama geometry split into q, k and v,
    and the fused gate/up projection with its SwiGLU epilogue."""
    rng = np.random.default_rng(61)
    T, dim = 4, 4096
    x = S.normal_bf16(rng, (T, dim))
    wqkv = S.normal_bf16(rng, (6144, dim), dim ** -0.5)
    ws = _ws(T, 28672)
    q = torch.empty((T, 4096), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((T, 1024), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((T, 1024), dtype=torch.bfloat16, device="cuda")
    # one workspace for both calls: the second one's tile counters must not be
    # the first one's partials
    P.c2kv_linear(to_dev(x), to_dev(wqkv), q, ws, P.C2KV_LINEAR_SPLIT3, y2=k, y3=v, split1=4096, split2=5120)
    ref = DO.linear(x, wqkv)
    check_rounded(q, ref[:, :4096], "q")
    check_rounded(k, ref[:, 4096:5120], "k")
    check_rounded(v, ref[:, 5120:], "v")
    wgu = S.normal_bf16(rng, (28672, dim), dim ** -0.5)
    m = torch.empty((T, 14336), dtype=torch.bfloat16, device="cuda")
    P.c2kv_linear(to_dev(x), to_dev(wgu), m, ws, P.C2KV_LINEAR_SWIGLU)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    check_rounded(m, DO.swiglu(x, wgu), "swiglu")


@pytest.mark.parametrize("n_feat", [512, 20480])
def test_swiglu_cluster_and_global_merge(n_feat):
    """SwiGLU on the two other splits: 8 tiles (clusters of 8 CTAs summing the
    gate/up partials in distributed shared memory) and 320 tiles (more than
    the CTAs: the even split with the global merge)."""
    rng = np.random.default_rng(n_feat)
    T, dim = 4, 4096
    x = S.normal_bf16(rng, (T, dim))
    wgu = S.normal_bf16(rng, (2 * n_feat, dim), dim ** -0.5)
    ws = _ws(T, 2 * n_feat)
    m = torch.empty((T, n_feat), dtype=torch.bfloat16, device="cuda")
    P.c2kv_linear(to_dev(x), to_dev(wgu), m, ws, P.C2KV_LINEAR_SWIGLU)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    check_rounded(m, DO.swiglu(x, wgu), f"swiglu F={n_feat}")


def test_split3_in_clusters():
    """A 3-tile q/k/v projection (clusters of 8 CTAs per tile) with split
    points inside the tiles' rows."""
    rng = np.random.default_rng(83)
    T, dim = 3, 4096
    x = S.normal_bf16(rng, (T, dim))
    w = S.normal_bf16(rng, (384, dim), dim ** -0.5)
    ws = _ws(T, 384)
    q = torch.empty((T, 200), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((T, 100), dtype=torch.bfloat16, device="cuda")
    v = torch.empty((T, 84), dtype=torch.bfloat16, device="cuda")
    P.c2kv_linear(to_dev(x), to_dev(w), q, ws, P.C2KV_LINEAR_SPLIT3, y2=k, y3=v, split1=200, split2=300)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    ref = DO.linear(x, w)
    check_rounded(q, ref[:, :200], "q")
    check_rounded(k, ref[:, 200:300], "k")
    check_rounded(v, ref[:, 300:], "v")


def test_rmsnorm():
    rng = np.random.default_rng(67)
    for T, dim in ((4, 4096), (3, 5120), (1, 64)):
        x = S.normal_bf16(rng, (T, dim), 3.0)
        w = S.bf16_bits(1.0 + 0.1 * rng.standard_normal(dim, dtype=np.float32))
        y = torch.empty((T, dim), dtype=torch.bfloat16, device="cuda")
        P.c2kv_rmsnorm(to_dev(x), to_dev(w), y, 1e-5)
        check_rounded(y, DO.rms_norm(x, w, 1e-5), f"rmsnorm {T}x{dim}")


def test_decoder_layer_llama_batch4():
    """One Llama-3.1-8B decoder layer at full size (seeded weights) decoding
    one token for each of 4 composed requests: every stage against the oracle
    on the GPU's own inputs to that stage, and the layer end to end."""
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    shape = S.LLAMA31_8B_MODEL
    specs = [(i, 300 + 212 * i, -(-(300 + 212 * i) // 4)) for i in range(6)]
    requests = [([0, 3, 5], None), ([1], None), ([2, 4], [1, 0]), ([5, 4, 3, 2, 1, 0], None)]
    sc = Scenario(g, 4, specs, requests, q_len=0, decode_steps=1)
    bt = sc.batch
    bt.compose()
    bt.reset_decode()
    wts = S.make_decoder_weights(g, shape, 1, 0xDEC0DE)
    w = wts["layers"][0]
    dev_w = {"layers": [{n: to_dev(a) for n, a in w.items()}]}
    model = P.DecoderModel(g, shape, dev_w, batch=4)
    rng = np.random.default_rng(71)
    x = S.normal_bf16(rng, (4, shape.dim))
    model.x.copy_(to_dev(x))
    model.layer(0, bt)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    # the oracle's layer on the same inputs and composed caches
    st = sc.oracle_store()
    kcs, vcs, starts = [], [], []
    for b, req in enumerate(sc.reqs):
        _, lt, kr, vr = O.compose(st, req.doc_ids, req.order, sc.k, g.rope_theta, layers=[0])
        kcs.append(kr[0])
        vcs.append(vr[0])
        starts.append(lt)
    x2, ref = DO.decoder_layer_decode(x, w, kcs, vcs, starts, g.rope_theta, 32, 8, shape.eps)
    # stage by stage, each on the GPU's own input to it
    q, k, v = to_bits(model.q), to_bits(model.k), to_bits(model.v)
    h_ref = DO.bf16(DO.rms_norm(x, w["attn_norm"], shape.eps))
    qkv = DO.linear(h_ref, w["qkv"])
    check_rounded(model.q, qkv[:, :4096], "q")
    check_rounded(model.k, qkv[:, 4096:5120], "k")
    check_rounded(model.v, qkv[:, 5120:], "v")
    for b in range(4):
        o_ref, _ = O.attend_new_tokens(q[b].reshape(1, 32, 128), k[b].reshape(1, 8, 128), v[b].reshape(1, 8, 128),
                                       kcs[b], vcs[b], starts[b], g.rope_theta)
        check_attention(model.att[b].reshape(1, 32, 128), o_ref, f"attention seq {b}")
    # x1 (overwritten on the GPU by the layer's output) from the GPU's attention
    x1 = DO.bf16(O.bf16_to_f64(x) + DO.linear(to_bits(model.att), w["o"]))
    check_rounded(model.h, DO.rms_norm(x1, w["mlp_norm"], shape.eps), "mlp norm")
    check_rounded(model.m, DO.swiglu(to_bits(model.h), w["gate_up"]), "swiglu")
    check_rounded(model.x, O.bf16_to_f64(x1) + DO.linear(to_bits(model.m), w["down"]), "down + residual")
    # end to end
    got = O.bf16_to_f64(to_bits(model.x))
    err = np.abs(got - O.bf16_to_f64(x2))
    assert err.max() <= 4e-2 and err.mean() <= 4e-3, (err.max(), err.mean())
    sc.close()
