"""Seeded random shapes of the linear layer through the C ABI against the
fp64 oracle: 1 to 256 tokens, K from 64 to 8192, 1 to 80 output tiles, and
every epilogue (store, residual add, q/k/v split at random points, SwiGLU).
The tile count against the CTAs decides the split -- clusters of 2, 4 or 8,
one whole tile per CTA, or the even split with the global merge -- so the
mix reaches each.  Same bar as the decoder tests: one bf16 rounding of an
fp32 sum, within 1 ulp of the exact value (or 2^-14 of the RMS)."""
import numpy as np
import pytest
import torch

import oracle.decoder_oracle as DO
import compressed_composable_kv_gb300 as P
from compressed_composable_kv_gb300 import synth as S
from gpu_util import to_dev
from test_gpu_decoder import check_rounded

pytestmark = pytest.mark.gpu


def _case(i: int):
    rng = np.random.default_rng(0x11E0 + i)
    tokens = int(rng.choice([1, 2, 3, 4, 7, 16, 17, int(rng.integers(18, 257))]))
    k_in = 64 * int(rng.integers(1, 129))
    tiles = int(rng.choice([1, 2, 3, 8, 13, 32, 48, int(rng.integers(1, 81))]))
    epi = int(rng.choice([P.C2KV_LINEAR_STORE, P.C2KV_LINEAR_ADD, P.C2KV_LINEAR_SPLIT3, P.C2KV_LINEAR_SWIGLU]))
    n_out = 128 * tiles
    if epi == P.C2KV_LINEAR_SPLIT3 and n_out < 3:
        epi = P.C2KV_LINEAR_STORE
    return tokens, k_in, n_out, epi, 0x11E0 + i


CASES = [_case(i) for i in range(32)]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_random_linear(i):
    tokens, k_in, n_out, epi, seed = CASES[i]
    rng = np.random.default_rng(seed)
    x = S.normal_bf16(rng, (tokens, k_in))
    w = S.normal_bf16(rng, (n_out, k_in), k_in ** -0.5)
    ws = torch.zeros(P.c2kv_linear_workspace_size(tokens, n_out), dtype=torch.uint8, device="cuda")
    P.c2kv_workspace_init(ws)
    xd, wd = to_dev(x), to_dev(w)
    ref = DO.linear(x, w)
    what = f"linear {tokens}x{k_in}x{n_out} epilogue {epi}"
    if epi == P.C2KV_LINEAR_SWIGLU:
        m = torch.empty((tokens, n_out // 2), dtype=torch.bfloat16, device="cuda")
        P.c2kv_linear(xd, wd, m, ws, P.C2KV_LINEAR_SWIGLU)
        torch.cuda.synchronize()
        assert P.c2kv_device_error() == P.C2KV_OK
        check_rounded(m, DO.swiglu(x, w), what)
    elif epi == P.C2KV_LINEAR_SPLIT3:
        s1 = int(rng.integers(1, n_out - 1))
        s2 = int(rng.integers(s1 + 1, n_out))
        q = torch.empty((tokens, s1), dtype=torch.bfloat16, device="cuda")
        k = torch.empty((tokens, s2 - s1), dtype=torch.bfloat16, device="cuda")
        v = torch.empty((tokens, n_out - s2), dtype=torch.bfloat16, device="cuda")
        P.c2kv_linear(xd, wd, q, ws, P.C2KV_LINEAR_SPLIT3, y2=k, y3=v, split1=s1, split2=s2)
        torch.cuda.synchronize()
        assert P.c2kv_device_error() == P.C2KV_OK
        check_rounded(q, ref[:, :s1], what + " q")
        check_rounded(k, ref[:, s1:s2], what + " k")
        check_rounded(v, ref[:, s2:], what + " v")
    elif epi == P.C2KV_LINEAR_ADD:
        r = S.normal_bf16(rng, (tokens, n_out))
        y = to_dev(r)
        P.c2kv_linear(xd, wd, y, ws, P.C2KV_LINEAR_ADD, residual=y)
        torch.cuda.synchronize()
        assert P.c2kv_device_error() == P.C2KV_OK
        from oracle.c2kv_oracle import bf16_to_f64
        check_rounded(y, ref + bf16_to_f64(r), what)
    else:
        y = torch.empty((tokens, n_out), dtype=torch.bfloat16, device="cuda")
        P.c2kv_linear(xd, wd, y, ws)
        torch.cuda.synchronize()
        assert P.c2kv_device_error() == P.C2KV_OK
        check_rounded(y, ref, what)
