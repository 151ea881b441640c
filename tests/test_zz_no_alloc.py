"""c2kv_attend_decode_noalloc: decode for callers that cannot allocate device
memory (plugins that get only a stream and tensors, serving loops that freeze
allocations at start-up).  Its split-K scratch is the library's fixed device
array; its output must match c2kv_attend_decode with a caller workspace, on
two calls in a row (the second reuses the array the first left behind).

Named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import compressed_composable_kv_gb300 as P
from compressed_composable_kv_gb300 import synth as S
from gpu_util import MAX_ABS, MEAN_ABS, Scenario, to_dev

pytestmark = pytest.mark.gpu


def _close(a: torch.Tensor, b: torch.Tensor):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, (d.max().item(), d.mean().item())


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    specs = [(i, 4000, 1000) for i in range(8)]   # 8000 slots: many key splits
    sc = Scenario(g, 4, specs, [(list(range(8)), None), (list(range(8)), [7, 1, 3, 0, 2, 6, 5, 4])],
                  q_len=0, decode_steps=1)
    bt = sc.batch
    bt.compose()
    bt.reset_decode()
    rng = np.random.default_rng(11)
    q = to_dev(S.normal_bf16(rng, (2, 32, 128)))
    kn = to_dev(S.normal_bf16(rng, (2, 8, 128)))
    vn = to_dev(S.normal_bf16(rng, (2, 8, 128)))
    ref = torch.empty_like(q)
    P.c2kv_attend_decode(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, bt.n_cached_dev,
                         bt.max_keys_decode, q, kn, vn, ref, bt.workspace)
    outs = []
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        P.c2kv_attend_decode_noalloc(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, bt.n_cached_dev,
                                     bt.max_keys_decode, q, kn, vn, o)
        outs.append(o)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    for o in outs:
        _close(o, ref)
    sc.close()


def test_noalloc_decode_rejects_bad_arguments_before_enqueueing():
    g = S.Geometry(1, 32, 8, 128, 5.0e5)
    sc = Scenario(g, 4, [(1, 400, 100)], [([1], None)], q_len=0, decode_steps=1)
    bt = sc.batch
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_attend_decode_noalloc(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, bt.n_cached_dev,
                                     bt.cap + 1, q, kn, kn, torch.empty_like(q))
    assert e.value.status == P.C2KV_EINVAL
    sc.close()
