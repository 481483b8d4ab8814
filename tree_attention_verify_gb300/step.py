"""One verification step of a fixed-shape generation sub-batch, with every output
and workspace buffer allocated once up front (so a step enqueues exactly four
kernels and allocates nothing):

    rd_pack_beams -> rd_tree_attention -> rd_greedy_accept -> rd_unpack

This is argument marshalling around the C ABI; all computation runs in librd.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (rd_greedy_accept, rd_greedy_accept_workspace_size, rd_pack_beams,
               rd_tree_attention, rd_tree_attention_workspace_size, rd_unpack)

KERNELS = ("rd_pack_beams", "rd_tree_attention", "rd_greedy_accept", "rd_unpack")


class VerifyStep:
    def __init__(self, B: int, W: int, L: int, Hq: int, Hkv: int, D: int, V: int, Dh: int,
                 max_ctx: int, device, P_max: Optional[int] = None):
        self.B, self.W, self.L, self.V, self.Dh = B, W, L, V, Dh
        self.P = W * L if P_max is None else P_max
        self.max_ctx = max_ctx
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        P, NW = self.P, (self.P + 31) // 32
        self.pk = dict(tokens=torch.empty(B, P, **i32), packer=torch.empty(B, P, **i32),
                       unpacker=torch.empty(B, W, L, **i32), mask=torch.empty(B, P, NW, **i32),
                       depth=torch.empty(B, P, **i32), packed_len=torch.empty(B, **i32))
        self.o = torch.empty(B, P, Hq, D, dtype=torch.bfloat16, device=dev)
        self.acc = dict(argmax=torch.empty(B, P, **i32), accept_len=torch.empty(B, W, **i32),
                        best_beam=torch.empty(B, **i32), n_accepted=torch.empty(B, **i32),
                        out_tokens=torch.empty(B, L, **i32))
        self.hidden_out = torch.empty(B, W, L, Dh, dtype=torch.bfloat16, device=dev)
        ws_a = rd_tree_attention_workspace_size(B, P, Hq, Hkv, D, max_ctx, dev)
        self.ws_attn = torch.zeros(ws_a, dtype=torch.uint8, device=dev) if ws_a else None
        self.ws_acc = torch.zeros(max(8, rd_greedy_accept_workspace_size(B, P, V)),
                                  dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, **i32)

    def __call__(self, beams, q, k_new, v_new, k_cache, v_cache, ctx_offsets, logits, hidden,
                 stream=None, events=None):
        """Enqueue the four kernels.  `events`, if given, is a list of 5 CUDA events
        recorded on the stream around the kernels (for per-kernel timing)."""
        s = torch.cuda.current_stream() if stream is None else stream
        ev = events
        if ev:
            ev[0].record(s)
        rd_pack_beams(beams, self.P, out=self.pk, dev_status=self.status, stream=s)
        if ev:
            ev[1].record(s)
        rd_tree_attention(q, k_new, v_new, k_cache, v_cache, ctx_offsets, self.pk["packed_len"],
                          self.pk["mask"], max_ctx=self.max_ctx, out=self.o,
                          workspace=self.ws_attn, dev_status=self.status, stream=s)
        if ev:
            ev[2].record(s)
        rd_greedy_accept(logits, beams, self.pk["unpacker"], self.pk["packed_len"], out=self.acc,
                         workspace=self.ws_acc, dev_status=self.status, stream=s)
        if ev:
            ev[3].record(s)
        rd_unpack(hidden, self.pk["unpacker"], out=self.hidden_out, dev_status=self.status,
                  stream=s)
        if ev:
            ev[4].record(s)
        return self.acc
