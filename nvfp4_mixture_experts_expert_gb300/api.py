"""Torch-side convenience layer over the C ABI: allocates outputs and
workspaces with torch on the current CUDA device and calls the binding.
No arithmetic of the method happens here."""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


def _round_up(x, m):
    return (x + m - 1) // m * m


def _u8(n, device):
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def quantize(x: torch.Tensor, gs: torch.Tensor | None = None, rows_padded: int | None = None, stream=None):
    """NVFP4-quantize the rows of a 2-D bf16 tensor.  Returns (fp4 [Rp, K/2] u8,
    sf (tile layout, Rp*K/16 bytes) u8, gs f32[1])."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, K = x.shape
    Rp = rows_padded if rows_padded is not None else _round_up(max(R, 1), 128)
    dev = x.device
    fp4 = torch.empty((Rp, K // 2), dtype=torch.uint8, device=dev)
    sf = _u8(Rp * K // 16, dev)
    gs_out = torch.empty(1, dtype=torch.float32, device=dev)
    ws = None
    wsb = 0
    if gs is None:
        wsb = B.nvfp4_quantize_workspace_size(1)
        ws = _u8(wsb, dev)
    B.nvfp4_quantize(x, R, K, x.stride(0), 0, 1, gs, gs_out, ws, wsb, fp4, sf, Rp, stream)
    return fp4, sf, gs_out


def quantize_groups(x: torch.Tensor, rows: int, K: int, ld_x: int, group_stride_x: int, groups: int,
                    gs: torch.Tensor | None = None, rows_padded: int | None = None, stream=None):
    """Quantize `groups` strided groups of rows of a bf16 buffer (see nvfp4_quantize)."""
    Rp = rows_padded if rows_padded is not None else _round_up(max(rows, 1), 128)
    dev = x.device
    fp4 = torch.empty((groups * Rp, K // 2), dtype=torch.uint8, device=dev)
    sf = _u8(groups * Rp * K // 16, dev)
    gs_out = torch.empty(groups, dtype=torch.float32, device=dev)
    ws = None
    wsb = 0
    if gs is None:
        wsb = B.nvfp4_quantize_workspace_size(groups)
        ws = _u8(wsb, dev)
    B.nvfp4_quantize(x, rows, K, ld_x, group_stride_x, groups, gs, gs_out, ws, wsb, fp4, sf, Rp, stream)
    return fp4, sf, gs_out


def quantize_expert_weights(w: torch.Tensor, gs: torch.Tensor | None = None, stream=None):
    """w: bf16 [E, N, K] (K contiguous, N % 128 == 0).  One global scale per expert
    (2688/amax of the expert unless gs is given).  Returns (fp4 [E, N, K/2],
    sf [E, N*K/16], gs [E])."""
    E, N, K = w.shape
    assert N % 128 == 0 and w.is_contiguous()
    fp4, sf, gs_out = quantize_groups(w, N, K, K, N * K, E, gs=gs, rows_padded=N, stream=stream)
    return fp4.view(E, N, K // 2), sf.view(E, N * K // 16), gs_out


def grouped_gemm(A, SFA, a_gs, Bw, SFB, b_gs, padded_offsets, counts, N, K, D, ldd, group_stride_d, stream=None):
    G = a_gs.numel()
    B.nvfp4_grouped_gemm(A, SFA, a_gs, Bw, SFB, b_gs, padded_offsets, counts, G, A.shape[0], N, K, D, ldd,
                         group_stride_d, stream)
    return D


@dataclass
class MoEWeights:
    w13: torch.Tensor      # u8 [E, 2I, H/2]
    w13_sf: torch.Tensor   # u8 [E, 2I*H/16]
    w13_gs: torch.Tensor   # f32 [E]
    w2: torch.Tensor       # u8 [E, H, I/2]
    w2_sf: torch.Tensor    # u8 [E, H*I/16]
    w2_gs: torch.Tensor    # f32 [E]

    @property
    def E(self):
        return self.w13.shape[0]

    @property
    def I(self):
        return self.w13.shape[1] // 2

    @property
    def H(self):
        return self.w2.shape[1]


def quantize_moe_weights(w13_bf16, w2_bf16, stream=None) -> MoEWeights:
    a = quantize_expert_weights(w13_bf16, stream=stream)
    b = quantize_expert_weights(w2_bf16, stream=stream)
    return MoEWeights(a[0], a[1], a[2], b[0], b[1], b[2])


class MoEForward:
    """Holds a workspace sized for (T, H, I, E, top_k) and runs nvfp4_moe_forward."""

    def __init__(self, T, H, I, E, top_k, device="cuda"):
        self.T, self.H, self.I, self.E, self.top_k = T, H, I, E, top_k
        self.ws_bytes = B.nvfp4_moe_workspace_size(T, H, I, E, top_k)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.layout = B.nvfp4_moe_workspace_layout(T, H, I, E, top_k)

    def __call__(self, hidden, logits, w: MoEWeights, a1_gs, a2_gs, gate_limit=10.0, up_limit=10.0, out=None,
                 stream=None, l1_output="bf16"):
        """a2_gs None: each expert's L2 activation scale is taken from this
        batch's own L1 output (read back with batch_l2_scales()), kept as bf16
        or (l1_output="fp8") as FP8 blocks until it is requantized."""
        if out is None:
            out = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=hidden.device)
        if l1_output == "fp8":
            if a2_gs is not None:
                raise ValueError("the FP8 L1 output applies when the L2 scales come from the batch (a2_gs None)")
            B.nvfp4_moe_forward_l1_fp8(hidden, logits, self.T, self.H, self.I, self.E, self.top_k, w.w13, w.w13_sf,
                                       w.w13_gs, w.w2, w.w2_sf, w.w2_gs, a1_gs, gate_limit, up_limit,
                                       self.workspace, self.ws_bytes, out, stream)
        elif l1_output == "bf16":
            B.nvfp4_moe_forward(hidden, logits, self.T, self.H, self.I, self.E, self.top_k, w.w13, w.w13_sf,
                                w.w13_gs, w.w2, w.w2_sf, w.w2_gs, a1_gs, a2_gs, gate_limit, up_limit,
                                self.workspace, self.ws_bytes, out, stream)
        else:
            raise ValueError(f"l1_output must be 'bf16' or 'fp8', not {l1_output!r}")
        return out

    def routed(self, hidden, topk_ids, topk_weights, experts_start, w: MoEWeights, a1_gs, a2_gs, gate_limit=10.0,
               up_limit=10.0, out=None, stream=None):
        """Forward with expert parallelism: global top-k ids (int32 [T, k]) and weights
        (f32 [T, k]) from the model's router; this layer holds experts
        [experts_start, experts_start + E)."""
        if out is None:
            out = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=hidden.device)
        B.nvfp4_moe_forward_routed(hidden, topk_ids, topk_weights, experts_start, self.T, self.H, self.I, self.E,
                                   self.top_k, w.w13, w.w13_sf, w.w13_gs, w.w2, w.w2_sf, w.w2_gs, a1_gs, a2_gs,
                                   gate_limit, up_limit, self.workspace, self.ws_bytes, out, stream)
        return out

    def calibrate(self, hidden, logits, w: MoEWeights, gate_limit=10.0, up_limit=10.0, stream=None):
        """Per-expert activation global scales (a1_gs, a2_gs) from this batch."""
        a1 = torch.empty(self.E, dtype=torch.float32, device=hidden.device)
        a2 = torch.empty(self.E, dtype=torch.float32, device=hidden.device)
        B.nvfp4_moe_calibrate(hidden, logits, self.T, self.H, self.I, self.E, self.top_k, w.w13, w.w13_sf,
                              w.w13_gs, gate_limit, up_limit, self.workspace, self.ws_bytes, a1, a2, stream)
        return a1, a2

    def calibrate_routed(self, hidden, topk_ids, topk_weights, experts_start, w: MoEWeights, gate_limit=10.0,
                         up_limit=10.0, stream=None):
        """The same scales from the model router's global top-k (int32 / f32
        [T, k]) for the experts [experts_start, experts_start + E) held here."""
        a1 = torch.empty(self.E, dtype=torch.float32, device=hidden.device)
        a2 = torch.empty(self.E, dtype=torch.float32, device=hidden.device)
        B.nvfp4_moe_calibrate_routed(hidden, topk_ids, topk_weights, experts_start, self.T, self.H, self.I, self.E,
                                     self.top_k, w.w13, w.w13_sf, w.w13_gs, gate_limit, up_limit, self.workspace,
                                     self.ws_bytes, a1, a2, stream)
        return a1, a2

    def batch_l2_scales(self):
        """The L2 global scales the last call with a2_gs None used (f32 [E])."""
        off = self.layout["calib"] + 4 * self.E
        return self.workspace[off:off + 4 * self.E].view(torch.float32)

    def status(self, stream=None, reset=False):
        """Device status word of the last call on this workspace (waits for the stream)."""
        return B.nvfp4_read_device_status(self.workspace, stream, reset)

    def view(self, name, dtype, count):
        """A view of one intermediate of the last call (see nvfp4_moe_workspace_layout)."""
        off = self.layout[name]
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype)


class SharedExpertForward:
    """The shared expert's NVFP4 SwiGLU FFN over every token (no routing), with
    its workspace; weights are one expert of quantize_moe_weights (E = 1)."""

    def __init__(self, T, H, I, device="cuda"):
        self.T, self.H, self.I = T, H, I
        self.ws_bytes = max(B.nvfp4_shared_expert_workspace_size(T, H, I), 256)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)

    def status(self, stream=None, reset=False):
        """Device status word of the last call on this workspace (waits for the stream)."""
        return B.nvfp4_read_device_status(self.workspace, stream, reset)

    def __call__(self, hidden, w: MoEWeights, a1_gs, a2_gs, gate_limit=10.0, up_limit=10.0, out=None, stream=None):
        if out is None:
            out = torch.empty((self.T, self.H), dtype=torch.bfloat16, device=hidden.device)
        B.nvfp4_shared_expert_forward(hidden, self.T, self.H, self.I, w.w13, w.w13_sf, w.w13_gs, w.w2, w.w2_sf,
                                      w.w2_gs, a1_gs, a2_gs, gate_limit, up_limit, self.workspace, self.ws_bytes,
                                      out, stream)
        return out


class HostPipeline:
    """Streams batches from pinned host memory through one MoEForward.

    submit(h_hidden, h_logits, h_out) enqueues, for one batch, the host->device
    copy of its hidden states and router logits, the forward, and the
    device->host copy of its output, on three CUDA streams with two device
    buffer sets: the upload of batch i+1 and the download of batch i-1 overlap
    the forward of batch i (the forwards themselves run in order on one stream,
    sharing the forward's workspace).  Host tensors must be pinned; a batch's
    h_out is complete once the event submit() returned has completed (or after
    synchronize()).  Copies are plain cudaMemcpyAsync through torch; no
    arithmetic happens here."""

    def __init__(self, fwd: MoEForward, weights: MoEWeights, a1_gs, a2_gs, gate_limit=10.0, up_limit=10.0,
                 device=None):
        device = torch.device(device) if device is not None else a1_gs.device
        self.fwd, self.w, self.a1_gs, self.a2_gs = fwd, weights, a1_gs, a2_gs
        self.gate_limit, self.up_limit = gate_limit, up_limit
        T, H, E = fwd.T, fwd.H, fwd.E
        self.d_hidden = [torch.empty((T, H), dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.d_logits = [torch.empty((T, E), dtype=torch.float32, device=device) for _ in range(2)]
        self.d_out = [torch.empty((T, H), dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.s_in = torch.cuda.Stream(device=device)
        self.s_comp = torch.cuda.Stream(device=device)
        self.s_out = torch.cuda.Stream(device=device)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]    # batch's inputs are on the device
        self.ev_comp = [torch.cuda.Event() for _ in range(2)]  # batch's forward has finished
        self.ev_out = [torch.cuda.Event() for _ in range(2)]   # batch's output is on the host
        self.count = 0
        cur = torch.cuda.current_stream(device)  # weights / scales made there come first
        for st in (self.s_in, self.s_comp, self.s_out):
            st.wait_stream(cur)

    @property
    def h2d_bytes(self):
        return self.d_hidden[0].numel() * 2 + self.d_logits[0].numel() * 4

    @property
    def d2h_bytes(self):
        return self.d_out[0].numel() * 2

    def submit(self, h_hidden, h_logits, h_out):
        b = self.count & 1
        # buffer set b was last read by the forward of batch count-2 (inputs)
        # and by the download of batch count-2 (output)
        self.s_in.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.s_in):
            self.d_hidden[b].copy_(h_hidden, non_blocking=True)
            self.d_logits[b].copy_(h_logits, non_blocking=True)
        self.ev_in[b].record(self.s_in)
        self.s_comp.wait_event(self.ev_in[b])
        self.s_comp.wait_event(self.ev_out[b])
        self.fwd(self.d_hidden[b], self.d_logits[b], self.w, self.a1_gs, self.a2_gs, self.gate_limit,
                 self.up_limit, out=self.d_out[b], stream=self.s_comp)
        self.ev_comp[b].record(self.s_comp)
        self.s_out.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.s_out):
            h_out.copy_(self.d_out[b], non_blocking=True)
        self.ev_out[b].record(self.s_out)
        self.count += 1
        return self.ev_out[b]

    def synchronize(self):
        for s in (self.s_in, self.s_comp, self.s_out):
            s.synchronize()
