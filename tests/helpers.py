"""Shared helpers of the test-suite: host<->device marshalling of the seeded
inputs, oracle-side references, and the comparison metrics."""
from __future__ import annotations

import numpy as np

from oracle import nvfp4_oracle as O
from nvfp4_mixture_experts_expert_gb300 import workloads as W


def rel_frob(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (d if d > 0 else 1.0))


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def bf16_dev(bits):
    """uint16 bf16 bit patterns (numpy) -> torch bf16 CUDA tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(arr):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def bf16_host(t):
    """torch bf16 tensor -> float32 numpy values."""
    import torch
    return t.detach().float().cpu().numpy()


def oracle_packed_rows(x, gs, rows_padded):
    """Oracle NVFP4 of the rows of x [R,K] with scalar gs: packed bytes [Rp,K/2],
    tile-layout scales [Rp*K/16], linear scales [R,K/16], nibbles [R,K]."""
    nib, s = O.quantize_blocks(x, gs)
    R, K = x.shape
    packed = np.zeros((rows_padded, K // 2), np.uint8)
    packed[:R] = O.pack_nibbles(nib)
    swz = O.assemble_scales(s, np.array([0, R]), np.array([0, rows_padded]))
    return packed, swz, s, nib


class OracleMoE:
    """Everything the oracle says about one MoE workload: quantized weights,
    activation global scales, routing, slots, the L1 input/outputs and out."""

    def __init__(self, wl, calib_rows=None, a1_gs=None, a2_gs=None):
        self.wl = wl
        self.hidden = W.bf16_bits_to_f32(wl.hidden)
        self.w13q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w13))
        self.w2q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w2))
        if a1_gs is None or a2_gs is None:
            a1, a2 = O.calibrate_activation_scales(self.hidden, wl.logits, wl.top_k, self.w13q,
                                                   wl.gate_limit, wl.up_limit, row_limit=calib_rows)
            self.a1_gs = a1 if a1_gs is None else a1_gs
            self.a2_gs = a2 if a2_gs is None else a2_gs
        else:
            self.a1_gs, self.a2_gs = a1_gs, a2_gs
        self.ids, self.w = O.route(wl.logits, wl.top_k)
        self.meta = O.sort_slots(self.ids, self.w, wl.E)

    def forward(self):
        return O.moe_forward(self.hidden, self.wl.logits, self.wl.top_k, self.w13q, self.w2q, self.a1_gs,
                             self.a2_gs, self.wl.gate_limit, self.wl.up_limit, return_intermediates=True)

    def slot_activations(self):
        """Oracle A1 (packed [P, H/2]) and its tile-layout scales over P rows."""
        H = self.wl.H
        P = self.meta["P"]
        nib = np.zeros((P, H), np.uint8)
        s = np.zeros((P, H // 16), np.uint8)
        for e in range(self.wl.E):
            lo = int(self.meta["offsets"][e])
            n = int(self.meta["counts"][e])
            if n:
                toks = self.meta["sorted_token_ids"][lo:lo + n]
                nib[lo:lo + n], s[lo:lo + n] = O.quantize_blocks(self.hidden[toks], self.a1_gs[e])
        swz = O.assemble_scales(s, np.array([0, P]), np.array([0, P]))
        return O.pack_nibbles(nib), swz

    def token_output(self, t):
        """Oracle output row of one token, computed on its own (for sampled checks)."""
        H = self.wl.H
        acc = np.zeros(H)
        for j in range(self.wl.top_k):
            e = int(self.ids[t, j])
            h = O.expert_l1(self.hidden[t:t + 1], self.a1_gs[e], self.w13q[0][e], self.w13q[1][e],
                            self.w13q[2][e], self.wl.gate_limit, self.wl.up_limit)
            Y = O.expert_l2(h, self.a2_gs[e], self.w2q[0][e], self.w2q[1][e], self.w2q[2][e])
            acc += self.w[t, j] * Y[0]
        return O.bf16_round(acc.astype(np.float32))
