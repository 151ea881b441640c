"""Request-batch runtime over the C ABI: owns the device caches, the length
arrays and the attention scratch of a batch of composed requests.

It only allocates device memory (torch) and sequences C-ABI calls; every
step of the path (composition, re-rotation, append, attention) runs in the
CUDA library.  C2KV explainer (paper-daily.com), section "pipeline: extract,
store, concatenate": compose the retrieved documents, append the question,
then generate.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

from . import binding as B


@dataclass
class RequestSpec:
    doc_ids: List[int]
    order: Optional[List[int]] = None


class RequestBatch:
    """Device state of `len(requests)` composed requests sharing one store."""

    def __init__(self, store: int, geom, requests: Sequence[RequestSpec], k: int, q_len: int,
                 decode_steps: int, device: str = "cuda", cap_multiple: int = 32, realign: bool = True):
        self.store, self.geom, self.k = store, geom, k
        # realign=False: the "no position re-alignment" ablation (documents
        # keep their extraction positions)
        self.compose_flags = 0 if realign else B.C2KV_COMPOSE_NO_REALIGN
        self.requests = list(requests)
        self.q_len, self.decode_steps = q_len, decode_steps
        self.batch = len(self.requests)
        L, H, D = geom.n_layers, geom.n_kv_heads, geom.head_dim
        self.n_slots, self.l_tot = [], []
        for r in self.requests:
            nt, ns = [], []
            for d in r.doc_ids:
                a, b, _ = B.c2kv_store_lookup(store, d)
                nt.append(a)
                ns.append(b)
            _, _, n, lt = B.c2kv_plan(nt, ns, r.order)
            self.n_slots.append(n)
            self.l_tot.append(lt)
        need = max(self.n_slots) + q_len + decode_steps
        self.cap = max(cap_multiple, -(-need // cap_multiple) * cap_multiple)
        self.k_caches = [torch.empty((L, H, self.cap, D), dtype=torch.bfloat16, device=device)
                         for _ in range(self.batch)]
        self.v_caches = [torch.empty_like(t) for t in self.k_caches]
        self.pos = [torch.full((self.cap,), -1, dtype=torch.int32, device=device)
                    for _ in range(self.batch)]
        tb = B.c2kv_rope_table_bytes(geom, self.cap)
        self.rope_tables = [torch.empty(tb // 4, dtype=torch.float32, device=device)
                            for _ in range(self.batch)]
        self.n_cached_dev = torch.zeros(self.batch, dtype=torch.int32, device=device)
        self.max_keys_decode = max(self.n_slots) + q_len + decode_steps
        ws = 256
        if q_len > 0:
            ws = max(ws, B.c2kv_attend_workspace_size(geom, self.batch, q_len, max(self.n_slots) + q_len))
        ws = max(ws, B.c2kv_attend_workspace_size(geom, self.batch, 1, self.max_keys_decode))
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=device)
        B.c2kv_workspace_init(self.workspace)
        self._dec_start = torch.tensor([n + q_len for n in self.n_slots], dtype=torch.int32)

    def compose(self, stream=None) -> None:
        self.compose_layers(0, self.geom.n_layers, stream)

    def compose_layers(self, layer_begin: int, layer_end: int, stream=None) -> None:
        """Compose layers [layer_begin, layer_end) of every request.  A call
        with layer_begin > 0 continues the composition of the call before it
        (C2KV_COMPOSE_CONTINUE): its copies follow that call's copies, so work
        enqueued in between on the earlier layers (the question prefill)
        overlaps them ("the problem": loading the cache dominates TTFT)."""
        flags = self.compose_flags | (B.C2KV_COMPOSE_CONTINUE if layer_begin > 0 else 0)
        for b, r in enumerate(self.requests):
            n, nxt = B.c2kv_compose_layers(self.store, r.doc_ids, r.order, self.k, flags, layer_begin,
                                           layer_end, self.k_caches[b], self.v_caches[b], self.cap,
                                           self.rope_tables[b], self.pos[b], stream)
            assert n == self.n_slots[b] and nxt == self.l_tot[b]

    def prefill(self, layer: int, q, k_new, v_new, out, stream=None) -> None:
        B.c2kv_attend_prefill(self.geom, layer, self.k_caches, self.v_caches, self.rope_tables, self.cap,
                              self.n_slots, q, k_new, v_new, out, self.workspace, stream)

    def reset_decode(self, stream=None) -> None:
        """Point the device lengths at the first decode step (after the question)."""
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            self.n_cached_dev.copy_(self._dec_start, non_blocking=True)

    def decode(self, layer: int, q, k_new, v_new, out, stream=None, overlap_previous: Optional[bool] = None) -> None:
        """One decode step of one layer.  By default a layer > 0 call may start
        while the previous kernel on the stream (this batch's decode of the
        layer before) finishes: see C2KV_DECODE_OVERLAP_PREVIOUS."""
        if overlap_previous is None:
            overlap_previous = layer > 0
        B.c2kv_attend_decode(self.geom, layer, self.k_caches, self.v_caches, self.rope_tables, self.cap,
                             self.n_cached_dev, self.max_keys_decode, q, k_new, v_new, out, self.workspace,
                             stream, B.C2KV_DECODE_OVERLAP_PREVIOUS if overlap_previous else 0)

    def advance(self, stream=None) -> None:
        B.c2kv_seq_advance(self.n_cached_dev, 1, stream)


class DecoderModel:
    """A synthetic-weight decoder stack around a RequestBatch's attention, on
    the device (C2KV explainer, section "the problem", Fig. 1: the decode rate
    of the whole model).  The layer is the Llama-3 one (no biases):
        h = rmsnorm(x) * w_attn; q | k | v = h W_qkv^T (split by the epilogue)
        x += attention(q, k, v) W_o^T          (the batch's composed caches)
        h = rmsnorm(x) * w_mlp;  x += (silu(h W_g^T) * h W_u^T) W_d^T
    then rmsnorm and the LM head.  Every step is a C-ABI call; launches after
    the first may overlap the tail of the one before (programmatic dependent
    launch): each kernel touches its activations only after the previous one
    has finished.

    weights: dict as synth.make_decoder_weights, values device bf16 tensors.
    """

    def __init__(self, geom, shape, weights: dict, batch: int, device: str = "cuda"):
        self.geom, self.shape, self.w = geom, shape, weights
        self.batch = batch
        d = geom.head_dim
        self.nq, self.nkv = geom.n_q_heads * d, geom.n_kv_heads * d
        nb, dim, F = batch, shape.dim, shape.ffn
        bf = torch.bfloat16

        def buf(*sz):
            return torch.zeros(sz, dtype=bf, device=device)

        self.x, self.h = buf(nb, dim), buf(nb, dim)
        self.q, self.k, self.v = buf(nb, self.nq), buf(nb, self.nkv), buf(nb, self.nkv)
        self.att, self.m = buf(nb, self.nq), buf(nb, F)
        has_head = "lm_head" in weights
        self.logits = buf(nb, shape.vocab) if has_head else None
        widest = max(self.nq + 2 * self.nkv, 2 * F, dim, shape.vocab if has_head else 0)
        self.workspace = torch.zeros(B.c2kv_linear_workspace_size(nb, widest), dtype=torch.uint8, device=device)
        B.c2kv_workspace_init(self.workspace)

    def layer(self, l: int, rb: "RequestBatch", stream=None) -> None:
        w = self.w["layers"][l]
        ov = B.C2KV_LINEAR_OVERLAP_PREVIOUS
        eps = self.shape.eps
        B.c2kv_rmsnorm(self.x, w["attn_norm"], self.h, eps, stream, ov)
        B.c2kv_linear(self.h, w["qkv"], self.q, self.workspace, B.C2KV_LINEAR_SPLIT3, y2=self.k, y3=self.v,
                       split1=self.nq, split2=self.nq + self.nkv, stream=stream, flags=ov)
        rb.decode(l, self.q, self.k, self.v, self.att, stream, overlap_previous=True)
        B.c2kv_linear(self.att, w["o"], self.x, self.workspace, B.C2KV_LINEAR_ADD, residual=self.x,
                       stream=stream, flags=ov)
        B.c2kv_rmsnorm(self.x, w["mlp_norm"], self.h, eps, stream, ov)
        B.c2kv_linear(self.h, w["gate_up"], self.m, self.workspace, B.C2KV_LINEAR_SWIGLU, stream=stream,
                       flags=ov)
        B.c2kv_linear(self.m, w["down"], self.x, self.workspace, B.C2KV_LINEAR_ADD, residual=self.x,
                       stream=stream, flags=ov)

    def decode_step(self, rb: "RequestBatch", stream=None) -> None:
        """One answer token per sequence: every layer, the LM head (if the
        weights have one), then the batch's lengths advance.  x holds the
        step's input embeddings and is updated in place."""
        for l in range(len(self.w["layers"])):
            self.layer(l, rb, stream)
        if self.logits is not None:
            B.c2kv_rmsnorm(self.x, self.w["final_norm"], self.h, self.shape.eps, stream,
                            B.C2KV_LINEAR_OVERLAP_PREVIOUS)
            B.c2kv_linear(self.h, self.w["lm_head"], self.logits, self.workspace, stream=stream,
                           flags=B.C2KV_LINEAR_OVERLAP_PREVIOUS)
        rb.advance(stream)

    def linears_only(self, stream=None) -> None:
        """The step's linear layers and norms without the attention (their
        own weight-streaming rate, for the roofline)."""
        ov = B.C2KV_LINEAR_OVERLAP_PREVIOUS
        eps = self.shape.eps
        for w in self.w["layers"]:
            B.c2kv_rmsnorm(self.x, w["attn_norm"], self.h, eps, stream, ov)
            B.c2kv_linear(self.h, w["qkv"], self.q, self.workspace, B.C2KV_LINEAR_SPLIT3, y2=self.k,
                           y3=self.v, split1=self.nq, split2=self.nq + self.nkv, stream=stream, flags=ov)
            B.c2kv_linear(self.att, w["o"], self.x, self.workspace, B.C2KV_LINEAR_ADD, residual=self.x,
                           stream=stream, flags=ov)
            B.c2kv_rmsnorm(self.x, w["mlp_norm"], self.h, eps, stream, ov)
            B.c2kv_linear(self.h, w["gate_up"], self.m, self.workspace, B.C2KV_LINEAR_SWIGLU, stream=stream,
                           flags=ov)
            B.c2kv_linear(self.m, w["down"], self.x, self.workspace, B.C2KV_LINEAR_ADD, residual=self.x,
                           stream=stream, flags=ov)
        if self.logits is not None:
            B.c2kv_rmsnorm(self.x, self.w["final_norm"], self.h, self.shape.eps, stream, ov)
            B.c2kv_linear(self.h, self.w["lm_head"], self.logits, self.workspace, stream=stream, flags=ov)

    def weight_bytes(self) -> int:
        n = sum(t.numel() for w in self.w["layers"] for t in w.values())
        if self.logits is not None:
            n += self.w["lm_head"].numel() + self.w["final_norm"].numel()
        return 2 * n
