"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/c2kv.h declares, and its host-side logic (planner, argument
checks, scratch sizing) behaves; no compute call is made."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle.c2kv_oracle as O
from compressed_composable_kv_gb300 import build
from compressed_composable_kv_gb300 import synth as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def P():
    build.build_library()
    import compressed_composable_kv_gb300 as pkg
    pkg.load_library()
    return pkg


def declared_functions():
    text = open(os.path.join(ROOT, "include", "c2kv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return sorted(set(re.findall(r"\b(c2kv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["c2kv_store_create", "c2kv_store_segments", "c2kv_compose", "c2kv_attend_prefill",
              "c2kv_attend_decode", "c2kv_attend_masked", "c2kv_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(P):
    lib = ctypes.CDLL(build.LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert P.c2kv_version().startswith("c2kv-gb300")


def test_binding_covers_every_declared_symbol(P):
    import compressed_composable_kv_gb300.binding as bnd
    for n in declared_functions():
        assert n in bnd._SIGNATURES, n


def test_plan_matches_oracle_positions(P):
    rng = np.random.default_rng(1)
    for _ in range(50):
        k = int(rng.choice([1, 4, 16]))
        n = int(rng.integers(1, 9))
        lens = [int(x) for x in rng.integers(1, 300, n)]
        slots = [O.slot_count(x, k) for x in lens]
        order = None if rng.random() < 0.3 else [int(x) for x in rng.permutation(n)]
        ss, po, total, l_tot = P.c2kv_plan(lens, slots, order)
        seq = O.composed_order(list(range(n)), order)
        pos, lt = O.composed_positions([lens[i] for i in seq], [slots[i] for i in seq], k)
        assert total == len(pos) and l_tot == lt
        for c, d in enumerate(seq):
            first = pos[ss[c]]
            assert first == O.extraction_slot_position(0, lens[d], k) + po[c]
            assert pos[ss[c] + slots[d] - 1] == po[c] + lens[d] - 1


@pytest.mark.parametrize("lens,slots,order", [
    ([4, 4], [1, 1], [0, 0]),        # not a permutation
    ([4, 4], [1, 1], [0, 2]),        # index out of range
    ([4, 0], [1, 1], None),          # empty document
    ([4, 4], [5, 1], None),          # more slots than tokens
    ([2**30, 2**30], [1, 1], None),  # position overflow
])
def test_plan_rejects_bad_input(P, lens, slots, order):
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_plan(lens, slots, order)
    assert e.value.status == P.C2KV_EINVAL
    assert P.c2kv_last_error()


def test_plan_empty(P):
    assert P.c2kv_plan([], [], None) == ([], [], 0, 0)


def test_workspace_sizing(P):
    g = S.LLAMA31_8B
    assert P.c2kv_attend_workspace_size(g, 1, 1, 8257) > 0
    assert P.c2kv_attend_workspace_size(g, 0, 1, 100) == 0
    bad = S.Geometry(32, 32, 8, 96, 5e5)
    assert P.c2kv_attend_workspace_size(bad, 1, 1, 100) == 0
    # more keys never needs fewer bytes
    sizes = [P.c2kv_attend_workspace_size(g, 4, 1, n) for n in (33, 1000, 8000, 33000)]
    assert sizes == sorted(sizes)
    assert P.c2kv_masked_extra_bytes(S.TINY, 15) >= 2 * 2 * 15 * 64 * 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_store_create_fails_cleanly_without_gpu(P):
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_store_create(S.TINY, 1 << 20)
    assert e.value.status in (P.C2KV_ECUDA, P.C2KV_ENOMEM)


def test_geometry_validation(P):
    for g in [S.Geometry(1, 6, 4, 64, 1e4), S.Geometry(1, 4, 2, 80, 1e4), S.Geometry(1, 4, 2, 64, 0.5)]:
        with pytest.raises(P.C2KVError) as e:
            P.c2kv_store_create(g, 0)
        assert e.value.status == P.C2KV_EINVAL


def test_store_file_and_test_hook_arguments_are_checked_on_the_host(P, tmp_path):
    """Null stores and negative counts are rejected before any CUDA call."""
    lib = P.load_library()
    assert lib.c2kv_store_save(None, os.fsencode(str(tmp_path / "x"))) == P.C2KV_EINVAL
    assert lib.c2kv_store_load(None, os.fsencode(str(tmp_path / "x"))) == P.C2KV_EINVAL
    with pytest.raises(P.C2KVError) as e:
        P.c2kv_test_expire_next_waits(-1)
    assert e.value.status == P.C2KV_EINVAL
    P.c2kv_test_expire_next_waits(0)
    assert P.STATUS_NAMES[P.C2KV_EIO] == "C2KV_EIO"



def test_kernel_launch_counter_is_host_only(P):
    """The launch counter reads without a GPU, counts nothing when nothing was
    launched, and rejects a null pointer."""
    assert P.c2kv_kernel_launches() == P.c2kv_kernel_launches() >= 0
    assert P.load_library().c2kv_kernel_launches(None) == P.C2KV_EINVAL


def test_masked_attention_arguments_are_checked_on_the_host(P):
    """Mask kinds and their size rules are checked before any pointer or CUDA
    call: an unknown mask, slots under the causal mask and k < 1 under the
    structured or anchor mask are rejected; a valid call then fails only on
    its null pointers."""
    lib = P.load_library()
    g = ctypes.byref(P.as_geometry(S.TINY))
    null = [None] * 5

    def call(mask, n_doc, n_slot, k):
        st = lib.c2kv_attend_masked(g, mask, n_doc, n_slot, k, *null[:4], null[4], 0, None)
        return st, P.c2kv_last_error()

    assert call(3, 8, 2, 4) == (P.C2KV_EINVAL, "unknown mask")
    assert call(P.C2KV_MASK_CAUSAL, 8, 2, 1)[1] == "causal mask takes n_slot = 0"
    for m in (P.C2KV_MASK_STRUCTURED, P.C2KV_MASK_ANCHOR):
        assert call(m, 8, 2, 0) == (P.C2KV_EINVAL, "k must be >= 1")
        assert call(m, 0, 2, 4)[1] == "need n_doc >= 1 and n_slot >= 0"
        assert call(m, 8, 2, 4) == (P.C2KV_EINVAL, "null pointer")


def test_store_segment_arrays_are_checked_by_the_binding(P, monkeypatch):
    """Host segments must be arrays of 2-byte elements of exactly the size the
    store's geometry gives (a converted temporary or a short array would be
    read past its end).  The null handle stands in for a store, so a check
    that let a bad array through would end in C2KV_EINVAL, not a read."""
    import compressed_composable_kv_gb300.binding as bnd
    g = S.TINY
    monkeypatch.setitem(bnd._STORE_GEOMETRY, 0, bnd.as_geometry(g))
    good = np.zeros((g.n_layers, g.n_kv_heads, 2, g.head_dim), np.uint16)
    bad = [
        [good.tolist()],                              # a list: would be converted into a temporary
        [good.astype(np.uint8)],                      # 1-byte elements
        [good[:, :, :1]],                             # one slot short of n_slots = 2
        [np.asfortranarray(good.transpose(3, 2, 1, 0))],   # not C-contiguous
        [torch.zeros(good.shape, dtype=torch.float32)],    # 4-byte elements
    ]
    for ks in bad:
        with pytest.raises(ValueError):
            P.c2kv_store_segments(0, [1], [8], [2], 4, ks, [good])
    with pytest.raises(ValueError):
        P.c2kv_store_segments(0, [1, 2], [8], [2], 4, [good], [good])   # lengths disagree
    with pytest.raises(P.C2KVError) as e:   # well-formed arrays reach the C side
        P.c2kv_store_segments(0, [1], [8], [2], 4, [good], [torch.from_numpy(good.view(np.int16))])
    assert e.value.status == P.C2KV_EINVAL


def test_device_buffer_sizes_are_checked_by_the_binding(P, monkeypatch):
    """The C side sees only pointers, so the binding checks every buffer
    against the sizes the call implies before anything is launched: one
    token short, a cache of too few rows or a table for too few rows raise
    ValueError (CPU tensors stand in: the size check comes first)."""
    import compressed_composable_kv_gb300.binding as bnd
    g = S.TINY
    Hq, Hkv, d, L = g.n_q_heads, g.n_kv_heads, g.head_dim, g.n_layers
    bf = torch.bfloat16
    N = 10
    short = torch.zeros((N - 1, Hq, d), dtype=bf)
    kv = torch.zeros((N, Hkv, d), dtype=bf)
    with pytest.raises(ValueError, match="q holds"):
        P.c2kv_attend_masked(g, P.C2KV_MASK_ANCHOR, 8, 2, 4, short, kv, kv, short, torch.zeros(16, dtype=torch.uint8))
    cap = 32
    cache = torch.zeros((L, Hkv, cap - 1, d), dtype=bf)       # one row short
    tab = torch.zeros(P.c2kv_rope_table_bytes(g, cap), dtype=torch.uint8)
    q1, k1 = torch.zeros((1, Hq, d), dtype=bf), torch.zeros((1, Hkv, d), dtype=bf)
    n_dev = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="k_caches"):
        P.c2kv_attend_decode(g, 0, [cache], [cache], [tab], cap, n_dev, 8, q1, k1, k1, q1, None)
    with pytest.raises(ValueError, match="k_caches"):
        P.c2kv_attend_decode_noalloc(g, 0, [cache], [cache], [tab], cap, n_dev, 8, q1, k1, k1, q1)
    good = torch.zeros((L, Hkv, cap, d), dtype=bf)
    with pytest.raises(ValueError, match="rope_tables"):
        P.c2kv_attend_decode(g, 0, [good], [good], [tab[:-16]], cap, n_dev, 8, q1, k1, k1, q1, None)
    with pytest.raises(ValueError, match="n_cached"):
        P.c2kv_attend_prefill(g, 0, [good], [good], [tab], cap, [0, 0], q1[None], k1[None], k1[None],
                              q1[None], None)
    with pytest.raises(ValueError, match="out holds"):
        P.c2kv_attend_prefill(g, 0, [good], [good], [tab], cap, [0], q1[None], k1[None], k1[None],
                              torch.zeros((1, 2, Hq, d), dtype=bf), None)
    with pytest.raises(ValueError, match="table_out"):
        P.c2kv_rope_table(g, torch.zeros(cap, dtype=torch.int32), tab[:-16])
    monkeypatch.setitem(bnd._STORE_GEOMETRY, 0, bnd.as_geometry(g))
    with pytest.raises(ValueError, match="rope_table"):
        P.c2kv_compose(0, [1], None, 4, good, good, cap, tab[:-16])
    with pytest.raises(ValueError, match="pos_dev_out"):
        P.c2kv_compose_layers(0, [1], None, 4, 0, 0, 1, good, good, cap, tab, torch.zeros(cap - 1, dtype=torch.int32))


def test_decode_scratch_fits_the_fixed_noalloc_array(P):
    """c2kv_attend_decode_noalloc keeps its scratch in a fixed 4 MiB device
    array and rejects a decode that would need more.  For every supported
    geometry on a 152-SM GPU (the sizing used without a GPU) the one-token
    scratch is far below that: two partial slots per SM plus per-unit
    counters at head_dim 128, at most one split per SM at head_dim 64."""
    limit = 4 << 20
    worst = 0
    for d in (64, 128):
        for grp in (1, 2, 4, 5, 8):
            for hkv in (1, 8, 1024 // (d // 16)):
                g = S.Geometry(1, hkv * grp, hkv, d, 1.0e4)
                for batch in (1, 4, 16):
                    for keys in (1, 1000, 131072, 1 << 22):
                        need = P.c2kv_attend_workspace_size(g, batch, 1, keys)
                        assert 0 < need
                        worst = max(worst, need)
    assert worst <= limit // 2, worst


def test_linear_and_rmsnorm_host_checks(P):
    """c2kv_linear / c2kv_rmsnorm reject bad shapes before touching the GPU;
    the linear workspace holds the fixed counter region plus two partial
    tiles per SM."""
    import compressed_composable_kv_gb300.binding as bnd
    lib = bnd.load_library()
    ws = ctypes.c_void_p(16)
    bad = [(0, 4096, 6144), (257, 4096, 6144), (4, 100, 6144), (4, 4096, 100), (4, 4096, 128 * 8193)]
    for tokens, k_in, n_out in bad:
        st = lib.c2kv_linear(ctypes.c_void_p(16), tokens, k_in, ctypes.c_void_p(16), n_out, 0, None,
                             ctypes.c_void_p(16), None, None, 0, 0, ws, 1 << 30, 0, None)
        assert st == P.C2KV_EINVAL, (tokens, k_in, n_out)
    st = lib.c2kv_linear(ctypes.c_void_p(16), 4, 4096, ctypes.c_void_p(16), 6144, P.C2KV_LINEAR_SPLIT3, None,
                         ctypes.c_void_p(16), None, None, 4096, 5120, ws, 1 << 30, 0, None)
    assert st == P.C2KV_EINVAL      # y2 / y3 missing
    st = lib.c2kv_linear(ctypes.c_void_p(16), 4, 4096, ctypes.c_void_p(16), 6144, 0, None,
                         ctypes.c_void_p(16), None, None, 0, 0, ws, 100, 0, None)
    assert st == P.C2KV_EINVAL and b"workspace" in lib.c2kv_last_error()
    assert lib.c2kv_rmsnorm(ctypes.c_void_p(16), 4, 100, ctypes.c_void_p(16), ctypes.c_float(1e-5),
                            ctypes.c_void_p(16), 0, None) == P.C2KV_EINVAL
    assert P.c2kv_linear_workspace_size(4, 6144) == 8192 * 4 + 2 * 304 * 16 * 128 * 4
    assert P.c2kv_linear_workspace_size(0, 6144) == 0
