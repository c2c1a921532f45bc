"""ctypes binding of libnvfp4moe (include/nvfp4moe.h): same names as the C ABI.

Argument marshalling only.  Tensor arguments may be torch tensors (their
device pointer is passed) or plain integers (device addresses); every
computation happens in the library's CUDA kernels.  A non-zero status raises
Nvfp4Error carrying the library's one-line reason.  Importing this module
fails loudly when the shared library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnvfp4moe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "nvfp4moe.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

c_i64 = ctypes.c_int64
c_int = ctypes.c_int
c_ptr = ctypes.c_void_p
c_size = ctypes.c_size_t
c_float = ctypes.c_float

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_UNSUPPORTED = 2
NVFP4_ERR_WORKSPACE = 3
NVFP4_ERR_CUDA = 4
NVFP4_ERR_DEVICE = 5
NVFP4_ERR_DEVICE_TIMEOUT = 6


class Nvfp4Error(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"nvfp4 status {status}: {msg}")
        self.status = status


class MoeLayout(ctypes.Structure):
    _fields_ = [(n, c_size) for n in (
        "status", "topk_ids", "topk_w", "block_counts", "counts", "offsets", "meta", "tile_expert",
        "sorted_token_ids", "row_weight", "inverse", "a1", "sfa1", "a2", "sfa2", "y", "h", "calib", "tile_done",
        "total")] + [
        ("capacity", c_i64), ("route_blocks", c_i64)]


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_lib_version = _sig("nvfp4_version", c_int, [])
_status_string = _sig("nvfp4_status_string", ctypes.c_char_p, [c_int])
_last_error = _sig("nvfp4_last_error", ctypes.c_char_p, [])
_quantize_ws = _sig("nvfp4_quantize_workspace_size", c_size, [c_int])
_quantize = _sig("nvfp4_quantize", c_int, [c_ptr, c_i64, c_i64, c_i64, c_i64, c_int, c_ptr, c_ptr, c_ptr, c_size,
                                           c_ptr, c_ptr, c_i64, c_ptr])
_quantize_no_alloc = _sig("nvfp4_quantize_no_alloc", c_int, [c_ptr, c_i64, c_i64, c_i64, c_i64, c_int, c_ptr,
                                                             c_ptr, c_ptr, c_i64, c_ptr])
_assemble = _sig("nvfp4_assemble_scales", c_int, [c_ptr, c_i64, c_ptr, c_ptr, c_int, c_i64, c_ptr, c_ptr])
_gemm = _sig("nvfp4_grouped_gemm", c_int, [c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_int, c_i64,
                                           c_i64, c_i64, c_ptr, c_i64, c_i64, c_ptr])
_gemm_stall = _sig("nvfp4_debug_gemm_stall", c_int, [c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_int, c_i64,
                                                      c_i64, c_i64, c_ptr, c_i64, c_int, c_ptr])
_moe_ws = _sig("nvfp4_moe_workspace_size", c_size, [c_i64, c_i64, c_i64, c_int, c_int])
_moe_layout = _sig("nvfp4_moe_workspace_layout", c_int, [c_i64, c_i64, c_i64, c_int, c_int,
                                                         ctypes.POINTER(MoeLayout)])
_moe_forward = _sig("nvfp4_moe_forward", c_int, [c_ptr, c_ptr, c_i64, c_i64, c_i64, c_int, c_int, c_ptr, c_ptr,
                                                 c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_float, c_float, c_ptr,
                                                 c_size, c_ptr, c_ptr])
_moe_forward_l1_fp8 = _sig("nvfp4_moe_forward_l1_fp8", c_int, [c_ptr, c_ptr, c_i64, c_i64, c_i64, c_int, c_int,
                                                               c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr,
                                                               c_float, c_float, c_ptr, c_size, c_ptr, c_ptr])
_moe_forward_routed = _sig("nvfp4_moe_forward_routed", c_int, [c_ptr, c_ptr, c_ptr, ctypes.c_int32, c_i64, c_i64,
                                                               c_i64, c_int, c_int, c_ptr, c_ptr, c_ptr, c_ptr,
                                                               c_ptr, c_ptr, c_ptr, c_ptr, c_float, c_float, c_ptr,
                                                               c_size, c_ptr, c_ptr])
_se_ws = _sig("nvfp4_shared_expert_workspace_size", c_size, [c_i64, c_i64, c_i64])
_se_forward = _sig("nvfp4_shared_expert_forward", c_int, [c_ptr, c_i64, c_i64, c_i64, c_ptr, c_ptr, c_ptr, c_ptr,
                                                          c_ptr, c_ptr, c_ptr, c_ptr, c_float, c_float, c_ptr,
                                                          c_size, c_ptr, c_ptr])
_moe_calibrate = _sig("nvfp4_moe_calibrate", c_int, [c_ptr, c_ptr, c_i64, c_i64, c_i64, c_int, c_int, c_ptr,
                                                     c_ptr, c_ptr, c_float, c_float, c_ptr, c_size, c_ptr, c_ptr,
                                                     c_ptr])
_moe_calibrate_routed = _sig("nvfp4_moe_calibrate_routed", c_int, [c_ptr, c_ptr, c_ptr, ctypes.c_int32, c_i64,
                                                                     c_i64, c_i64, c_int, c_int, c_ptr, c_ptr,
                                                                     c_ptr, c_float, c_float, c_ptr, c_size, c_ptr,
                                                                     c_ptr, c_ptr])
_device_status = _sig("nvfp4_device_status", c_int, [ctypes.POINTER(c_int), c_int])
_read_status = _sig("nvfp4_read_device_status", c_int, [c_ptr, c_ptr, ctypes.POINTER(c_int), c_int])
_debug_stall = _sig("nvfp4_moe_set_debug_stall", c_int, [c_int])
_gemm_trace = _sig("nvfp4_debug_gemm_trace", c_int, [c_ptr, c_int, c_int, c_int])
_mma_rate = _sig("nvfp4_debug_mma_rate", c_int, [c_ptr, c_size, c_ptr, c_size, c_ptr, c_size, c_ptr, c_size, c_int,
                                                 c_int, c_int, c_int, c_ptr])
_stage_events = _sig("nvfp4_moe_set_stage_events", c_int, [ctypes.POINTER(c_ptr), c_int])
_moe_set_overlap = _sig("nvfp4_moe_set_overlap", c_int, [c_int, ctypes.POINTER(c_int)])
_gemm_set_cta_pair = _sig("nvfp4_gemm_set_cta_pair", c_int, [c_int, ctypes.POINTER(c_int)])
_moe_set_swap_l2 = _sig("nvfp4_moe_set_swap_l2", c_int, [c_int, ctypes.POINTER(c_int)])


def _p(t):
    """Device address of a torch tensor / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc):
    if rc != NVFP4_OK:
        raise Nvfp4Error(rc, _last_error().decode() or _status_string(rc).decode())


def declared_functions():
    """Names of the functions include/nvfp4moe.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_\w+)\s*\(", text)))


def nvfp4_version():
    return _lib_version()


def nvfp4_status_string(status):
    return _status_string(status).decode()


def nvfp4_last_error():
    return _last_error().decode()


def nvfp4_quantize_workspace_size(groups):
    return _quantize_ws(groups)


def nvfp4_quantize(x, rows, K, ld_x, group_stride_x, groups, gs, gs_out, workspace, workspace_bytes, fp4, sf,
                   rows_padded, stream=None):
    _check(_quantize(_p(x), rows, K, ld_x, group_stride_x, groups, _p(gs), _p(gs_out), _p(workspace),
                     workspace_bytes, _p(fp4), _p(sf), rows_padded, _stream(stream)))


def nvfp4_quantize_no_alloc(x, rows, K, ld_x, group_stride_x, groups, gs_out, fp4, sf, rows_padded, stream=None):
    """nvfp4_quantize with gs computed on the device and no workspace argument, for
    callers that cannot allocate device memory (see include/nvfp4moe.h)."""
    _check(_quantize_no_alloc(_p(x), rows, K, ld_x, group_stride_x, groups, _p(gs_out), _p(fp4), _p(sf),
                              rows_padded, _stream(stream)))


def nvfp4_assemble_scales(sf_linear, sf_cols, offsets, padded_offsets, groups, rows_capacity, sf_swizzled,
                          stream=None):
    _check(_assemble(_p(sf_linear), sf_cols, _p(offsets), _p(padded_offsets), groups, rows_capacity,
                     _p(sf_swizzled), _stream(stream)))


def nvfp4_grouped_gemm(A, SFA, a_gs, B, SFB, b_gs, padded_offsets, counts, groups, rows_capacity, N, K, D, ldd,
                       group_stride_d, stream=None):
    _check(_gemm(_p(A), _p(SFA), _p(a_gs), _p(B), _p(SFB), _p(b_gs), _p(padded_offsets), _p(counts), groups,
                 rows_capacity, N, K, _p(D), ldd, group_stride_d, _stream(stream)))


def nvfp4_debug_gemm_stall(A, SFA, a_gs, B, SFB, b_gs, padded_offsets, groups, rows_capacity, N, K, D, ldd,
                           timeout_ms, stream=None):
    _check(_gemm_stall(_p(A), _p(SFA), _p(a_gs), _p(B), _p(SFB), _p(b_gs), _p(padded_offsets), groups,
                       rows_capacity, N, K, _p(D), ldd, timeout_ms, _stream(stream)))


def nvfp4_moe_workspace_size(T, H, I, E, top_k):
    return _moe_ws(T, H, I, E, top_k)


def nvfp4_moe_workspace_layout(T, H, I, E, top_k):
    L = MoeLayout()
    _check(_moe_layout(T, H, I, E, top_k, ctypes.byref(L)))
    return {n: getattr(L, n) for n, _ in MoeLayout._fields_}


def nvfp4_moe_forward(hidden, router_logits, T, H, I, E, top_k, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, a1_gs,
                      a2_gs, gate_limit, up_limit, workspace, workspace_bytes, out, stream=None):
    _check(_moe_forward(_p(hidden), _p(router_logits), T, H, I, E, top_k, _p(w13), _p(w13_sf), _p(w13_gs),
                        _p(w2), _p(w2_sf), _p(w2_gs), _p(a1_gs), _p(a2_gs), gate_limit, up_limit,
                        _p(workspace), workspace_bytes, _p(out), _stream(stream)))


def nvfp4_moe_forward_l1_fp8(hidden, router_logits, T, H, I, E, top_k, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, a1_gs,
                             gate_limit, up_limit, workspace, workspace_bytes, out, stream=None):
    _check(_moe_forward_l1_fp8(_p(hidden), _p(router_logits), T, H, I, E, top_k, _p(w13), _p(w13_sf), _p(w13_gs),
                               _p(w2), _p(w2_sf), _p(w2_gs), _p(a1_gs), gate_limit, up_limit, _p(workspace),
                               workspace_bytes, _p(out), _stream(stream)))


def nvfp4_moe_forward_routed(hidden, topk_ids, topk_weights, experts_start, T, H, I, E, top_k, w13, w13_sf,
                             w13_gs, w2, w2_sf, w2_gs, a1_gs, a2_gs, gate_limit, up_limit, workspace,
                             workspace_bytes, out, stream=None):
    _check(_moe_forward_routed(_p(hidden), _p(topk_ids), _p(topk_weights), int(experts_start), T, H, I, E, top_k,
                               _p(w13), _p(w13_sf), _p(w13_gs), _p(w2), _p(w2_sf), _p(w2_gs), _p(a1_gs),
                               _p(a2_gs), gate_limit, up_limit, _p(workspace), workspace_bytes, _p(out),
                               _stream(stream)))


def nvfp4_shared_expert_workspace_size(T, H, I):
    return int(_se_ws(T, H, I))


def nvfp4_shared_expert_forward(hidden, T, H, I, w13, w13_sf, w13_gs, w2, w2_sf, w2_gs, a1_gs, a2_gs, gate_limit,
                                up_limit, workspace, workspace_bytes, out, stream=None):
    _check(_se_forward(_p(hidden), T, H, I, _p(w13), _p(w13_sf), _p(w13_gs), _p(w2), _p(w2_sf), _p(w2_gs),
                       _p(a1_gs), _p(a2_gs), gate_limit, up_limit, _p(workspace), workspace_bytes, _p(out),
                       _stream(stream)))


def nvfp4_moe_calibrate(hidden, router_logits, T, H, I, E, top_k, w13, w13_sf, w13_gs, gate_limit, up_limit,
                        workspace, workspace_bytes, a1_gs_out, a2_gs_out, stream=None):
    _check(_moe_calibrate(_p(hidden), _p(router_logits), T, H, I, E, top_k, _p(w13), _p(w13_sf), _p(w13_gs),
                          gate_limit, up_limit, _p(workspace), workspace_bytes, _p(a1_gs_out), _p(a2_gs_out),
                          _stream(stream)))


def nvfp4_moe_calibrate_routed(hidden, topk_ids, topk_weights, experts_start, T, H, I, E, top_k, w13, w13_sf,
                               w13_gs, gate_limit, up_limit, workspace, workspace_bytes, a1_gs_out, a2_gs_out,
                               stream=None):
    _check(_moe_calibrate_routed(_p(hidden), _p(topk_ids), _p(topk_weights), experts_start, T, H, I, E, top_k,
                                 _p(w13), _p(w13_sf), _p(w13_gs), gate_limit, up_limit, _p(workspace),
                                 workspace_bytes, _p(a1_gs_out), _p(a2_gs_out), _stream(stream)))


def nvfp4_device_status(reset=False):
    st = c_int(-1)
    _check(_device_status(ctypes.byref(st), 1 if reset else 0))
    return st.value


def nvfp4_read_device_status(workspace, stream=None, reset=False):
    """Status word of the last call that used this workspace (waits for `stream`)."""
    st = c_int(-1)
    _check(_read_status(_p(workspace), _stream(stream), ctypes.byref(st), 1 if reset else 0))
    return st.value


def nvfp4_debug_gemm_trace(buffer, stages=0, tiles=0, kind=-1):
    """Record the GEMM pipeline timeline of CTA 0 into `buffer` (int64 device tensor of
    (stages + tiles) * 8 words) for launches of epilogue `kind`; buffer None: off."""
    _check(_gemm_trace(_p(buffer), stages, tiles, kind))


def nvfp4_moe_set_debug_stall(timeout_ms):
    """> 0: following MoE forwards run their L1 GEMM with no operand loads (it times
    out after timeout_ms and records the timeout in the call's workspace); 0: off."""
    _check(_debug_stall(int(timeout_ms)))


def nvfp4_debug_mma_rate(A, a_bytes, SFA, sfa_bytes, B, b_bytes, SFB, sfb_bytes, shape, units, iters, flags=0,
                         stream=None):
    """The bare block-scaled FP4 MMA stream (see include/nvfp4moe.h); time it with events."""
    _check(_mma_rate(_p(A), a_bytes, _p(SFA), sfa_bytes, _p(B), b_bytes, _p(SFB), sfb_bytes, shape, units, iters,
                     flags, _stream(stream)))


def nvfp4_moe_set_overlap(enable):
    """1 (default): the L2 GEMM takes the L1 output m-tile by m-tile; 0: after
    the whole L1 GEMM.  Returns the previous setting."""
    prev = c_int(-1)
    _check(_moe_set_overlap(int(enable), ctypes.byref(prev)))
    return prev.value


def nvfp4_gemm_set_cta_pair(mode):
    """GEMM variant: 0 / False single CTAs, 1 / True CTA pairs, 2 pairs for the MoE L2
    GEMM only (default).  Returns the previous mode."""
    prev = c_int(-1)
    _check(_gemm_set_cta_pair(int(mode), ctypes.byref(prev)))
    return prev.value


def nvfp4_moe_set_swap_l2(enable):
    """1: the L2 GEMM of small batches runs with W2 tiles as the MMA's M operand
    and 64 slot rows as N; 0 (default): always slot-major.  Returns the previous setting."""
    prev = c_int(-1)
    _check(_moe_set_swap_l2(int(enable), ctypes.byref(prev)))
    return prev.value


def nvfp4_moe_set_stage_events(events):
    """events: list of 8 torch.cuda.Event (created with enable_timing) or None to switch off."""
    if not events:
        _check(_stage_events(None, 0))
        return
    handles = [e.cuda_event for e in events]
    if not all(handles):
        raise ValueError("stage events must have been recorded once (torch creates CUDA events lazily)")
    arr = (c_ptr * len(events))(*handles)
    _check(_stage_events(arr, len(events)))
