"""Seeded random shapes of the extraction-time attention (structured,
anchor-token and plain causal masks) through the C ABI against the fp64
oracle: documents of 1 to 1200 tokens, any number of extra tokens the mask
allows (the document's slot count, or none under the causal mask), k from 1
to 16, group sizes 1/2/4/5/8 and head_dim 64 and 128, so that the document /
slot boundary and the sink block fall anywhere inside the M and key tiles.
Same bar as the parity tests."""
import numpy as np
import pytest
import torch

import oracle.c2kv_oracle as O
import compressed_composable_kv_gb300 as P
from compressed_composable_kv_gb300 import synth as S
from gpu_util import check_attention, to_dev

pytestmark = pytest.mark.gpu


def _case(i: int):
    rng = np.random.default_rng(0x3A5C + i)
    G = int(rng.choice([1, 2, 4, 5, 8]))
    hkv = int(rng.choice([1, 2, 4]))
    d = int(rng.choice([64, 128]))
    mask = str(rng.choice(["structured", "anchor", "causal"]))
    n_doc = int(rng.choice([1, 2, int(rng.integers(3, 130)), int(rng.integers(130, 1200))], p=[0.1, 0.1, 0.4, 0.4]))
    k = int(rng.choice([1, 2, 3, 4, 8, 16]))
    n_slot = 0 if mask == "causal" else O.slot_count(n_doc, k)
    return S.Geometry(1, G * hkv, hkv, d, float(rng.choice([1.0e4, 5.0e5]))), mask, n_doc, n_slot, k, 0x3A5C + i


CASES = [_case(i) for i in range(32)]
CODES = {"structured": P.C2KV_MASK_STRUCTURED, "anchor": P.C2KV_MASK_ANCHOR, "causal": P.C2KV_MASK_CAUSAL}


@pytest.mark.parametrize("i", range(len(CASES)))
def test_random_masked(i):
    g, mask, n_doc, n_slot, k, seed = CASES[i]
    rng = np.random.default_rng(seed)
    N = n_doc + n_slot
    q = S.normal_bf16(rng, (N, g.n_q_heads, g.head_dim))
    kk = S.normal_bf16(rng, (N, g.n_kv_heads, g.head_dim))
    v = S.normal_bf16(rng, (N, g.n_kv_heads, g.head_dim))
    ws = torch.zeros(P.masked_workspace_bytes(g, N), dtype=torch.uint8, device="cuda")
    out = torch.empty((N, g.n_q_heads, g.head_dim), dtype=torch.bfloat16, device="cuda")
    P.c2kv_attend_masked(g, CODES[mask], n_doc, n_slot, k, to_dev(q), to_dev(kk), to_dev(v), out, ws)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    # with no extra tokens the structured mask is the plain causal one
    ref = O.masked_extraction_attention(q, kk, v, n_doc, n_slot, k, g.rope_theta,
                                        mask="structured" if mask == "causal" else mask)
    check_attention(out, ref, f"{mask} mask {n_doc}+{n_slot} k={k} G={g.group} d={g.head_dim}")
