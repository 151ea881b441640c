"""c2kv_attend_decode_noalloc: decode for callers that cannot allocate device
memory where they decode -- a plugin whose host framework hands it only a
stream and tensors and forbids allocating while it enqueues work, or a
serving loop that fixes every device allocation at start-up.  Its split-K
scratch is one fixed array in the library's own device memory.

Checked here: on two calls in a row (the second reuses the array the first
left behind) the output matches c2kv_attend_decode with a caller workspace
and the CPU oracle, and no device memory is allocated by the calls; bad
arguments are rejected before anything is enqueued.

Named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import compressed_composable_kv_gb300 as P
from compressed_composable_kv_gb300 import synth as S
from gpu_util import MAX_ABS, MEAN_ABS, Scenario, check_request, to_dev, upload

pytestmark = pytest.mark.gpu

LLAMA1 = S.Geometry(1, 32, 8, 128, 5.0e5)
QWEN1 = S.Geometry(1, 40, 8, 128, 1.0e6)

# (geometry, k, documents (id, tokens, slots), requests): one sequence of 8000
# slots (thread-block cluster merge), four of unequal lengths (partials merged
# through global memory), and the Qwen group of 5 heads
CASES = {
    "llama_b1_8000": (LLAMA1, 4, [(i, 4000, 1000) for i in range(8)], [(list(range(8)), [7, 1, 3, 0, 2, 6, 5, 4])]),
    "llama_b4_unequal": (LLAMA1, 4, [(i, 1000 + 700 * i, 250 + 175 * i) for i in range(6)],
                         [([0, 5, 2], None), ([1], None), ([3, 4], [1, 0]), ([5, 4, 3, 2, 1, 0], None)]),
    "qwen_g5_b2": (QWEN1, 16, [(i, 8000, 500) for i in range(4)], [([0, 1, 2, 3], None), ([3, 2], None)]),
}


def _close(a: torch.Tensor, b: torch.Tensor):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, (d.max().item(), d.mean().item())


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_decode_matches_oracle_and_workspace_decode_on_two_calls(case):
    g, k, specs, requests = CASES[case]
    sc = Scenario(g, k, specs, requests, q_len=0, decode_steps=1)
    w = S.Workload(case, g, k, len(requests), 0, 1, seed=0xC2D0)
    inputs = S.make_step_inputs(w)
    dev = upload(inputs)
    bt = sc.batch
    bt.compose()
    bt.reset_decode()
    q, kn, vn = dev["qd_pre"][0, 0], dev["kd_pre"][0, 0], dev["vd"][0, 0]
    ref = torch.empty_like(q)
    P.c2kv_attend_decode(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, bt.n_cached_dev,
                         bt.max_keys_decode, q, kn, vn, ref, bt.workspace)
    outs = [torch.full_like(q, float("nan")) for _ in range(3)]

    def call(o):
        P.c2kv_attend_decode_noalloc(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, bt.n_cached_dev,
                                     bt.max_keys_decode, q, kn, vn, o)

    call(outs[0])   # the first call on the device looks up the array's address
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    allocs0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    call(outs[1])
    call(outs[2])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across the calls"
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs0
    assert P.c2kv_device_error() == P.C2KV_OK
    for o in outs[1:]:
        _close(o, ref)
        # every call appends the same new key at the same row, so each output
        # is step 0 of the oracle's decode
        for b in range(len(requests)):
            check_request(sc, inputs, [], [[o]], b, layers=[0], steps=[0])
    sc.close()


def test_noalloc_decode_rejects_bad_arguments_before_enqueueing():
    g = LLAMA1
    sc = Scenario(g, 4, [(1, 400, 100)], [([1], None)], q_len=0, decode_steps=1)
    bt = sc.batch
    q = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(P.C2KVError) as e:   # max_keys beyond the cache
        P.c2kv_attend_decode_noalloc(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, bt.n_cached_dev,
                                     bt.cap + 1, q, kn, kn, out)
    assert e.value.status == P.C2KV_EINVAL
    # q that starts 2 bytes into its buffer (not 16-byte aligned)
    buf = torch.zeros(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    q_odd = buf[1:1 + q.numel()].view(q.shape)
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_attend_decode_noalloc(g, 0, bt.k_caches, bt.v_caches, bt.rope_tables, bt.cap, bt.n_cached_dev,
                                     8, q_odd, kn, kn, out)
    assert e.value.status == P.C2KV_EINVAL and "aligned" in str(e.value)
    torch.cuda.synchronize()
    assert P.c2kv_device_error() == P.C2KV_OK
    sc.close()
