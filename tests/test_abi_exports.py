"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
function include/nvfp4moe.h declares, and rejects bad arguments on the host
before touching a device (no compute call is made here)."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def binding():
    from nvfp4_mixture_experts_expert_gb300 import _build
    _build.build()
    from nvfp4_mixture_experts_expert_gb300 import binding as B
    return B


def test_every_declared_symbol_is_exported(binding):
    names = binding.declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(binding.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(binding):
    assert binding.nvfp4_version() >= 100
    for code in range(7):
        assert binding.nvfp4_status_string(code)


def test_workspace_layout_is_consistent(binding):
    T, H, I, E, k = 8192, 4096, 2048, 48, 6
    L = binding.nvfp4_moe_workspace_layout(T, H, I, E, k)
    assert L["capacity"] == 55296  # roundup(T*k + 127*E, 128)
    order = ["status", "topk_ids", "topk_w", "block_counts", "counts", "offsets", "meta", "tile_expert",
             "sorted_token_ids", "row_weight", "inverse", "a1", "sfa1", "a2", "sfa2", "y", "h", "calib", "tile_done"]
    offs = [L[n] for n in order]
    assert offs == sorted(offs) and all(o % 1024 == 0 for o in offs)
    assert L["status"] == 0  # the status word sits at byte 0 of the workspace
    assert L["sfa1"] - L["a1"] >= L["capacity"] * H // 2
    assert L["h"] - L["y"] >= L["capacity"] * H * 2
    assert L["calib"] - L["h"] >= L["capacity"] * I * 2
    assert L["total"] - L["tile_done"] >= L["capacity"] // 128 * 4
    assert binding.nvfp4_moe_workspace_size(T, H, I, E, k) == L["total"]


@pytest.mark.parametrize("args,code", [
    (dict(K=48), 1),          # K not a multiple of 64
    (dict(rows_padded=100), 1),
    (dict(groups=0), 1),
    (dict(ld_x=60), 1),
])
def test_quantize_rejects_bad_arguments_on_host(binding, args, code):
    kw = dict(x=16, rows=10, K=64, ld_x=64, group_stride_x=0, groups=1, gs=16, gs_out=None, workspace=None,
              workspace_bytes=0, fp4=16, sf=16, rows_padded=128)
    kw.update(args)
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_quantize(kw["x"], kw["rows"], kw["K"], kw["ld_x"], kw["group_stride_x"], kw["groups"],
                               kw["gs"], kw["gs_out"], kw["workspace"], kw["workspace_bytes"], kw["fp4"],
                               kw["sf"], kw["rows_padded"], stream=0)
    assert ei.value.status == code
    assert binding.nvfp4_last_error()


def test_gemm_and_moe_reject_unsupported_shapes(binding):
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_grouped_gemm(16, 16, 16, 16, 16, 16, 16, None, 1, 128, 204, 64, 16, 208, 0, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG  # N must be a multiple of 8
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_moe_forward(16, 16, 4, 4096, 2048, 48, 9, 16, 16, 16, 16, 16, 16, 16, 16, 10.0, 10.0,
                                  16, 1 << 30, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG
    with pytest.raises(binding.Nvfp4Error) as ei:  # workspace too small
        binding.nvfp4_moe_forward(16, 16, 4, 256, 128, 4, 2, 16, 16, 16, 16, 16, 16, 16, 16, 10.0, 10.0,
                                  256, 10, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_WORKSPACE


def test_gemm_variant_mode_setter(binding):
    """Host-only: the default mode pairs only the L2 GEMM (2); set returns the
    previous mode; an out-of-range mode is refused and leaves the mode alone."""
    prev = binding.nvfp4_gemm_set_cta_pair(0)
    try:
        assert prev == 2
        assert binding.nvfp4_gemm_set_cta_pair(1) == 0
        with pytest.raises(binding.Nvfp4Error) as ei:
            binding.nvfp4_gemm_set_cta_pair(3)
        assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG
        assert binding.nvfp4_gemm_set_cta_pair(1) == 1
    finally:
        binding.nvfp4_gemm_set_cta_pair(prev)


def test_routed_and_shared_expert_entries_check_arguments_on_host(binding):
    # routed forward: ids / weights required, sizes as the logit forward
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_moe_forward_routed(16, None, 16, 0, 4, 256, 128, 4, 2, 16, 16, 16, 16, 16, 16, 16, 16, 10.0,
                                         10.0, 256, 1 << 30, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_moe_forward_routed(16, 16, 16, 0, 4, 300, 128, 4, 2, 16, 16, 16, 16, 16, 16, 16, 16, 10.0,
                                         10.0, 256, 1 << 30, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_UNSUPPORTED
    # shared expert: H % 256, I % 128, workspace size and alignment
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_shared_expert_forward(16, 4, 300, 128, 16, 16, 16, 16, 16, 16, 16, 16, 10.0, 10.0, 256,
                                            1 << 30, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_UNSUPPORTED
    need = binding.nvfp4_shared_expert_workspace_size(4, 256, 128)
    assert need > 0
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_shared_expert_forward(16, 4, 256, 128, 16, 16, 16, 16, 16, 16, 16, 16, 10.0, 10.0, 256,
                                            need - 1, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_WORKSPACE
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_shared_expert_forward(16, 4, 256, 128, 16, 16, 16, 16, 16, 16, 16, 16, 10.0, 10.0, 16,
                                            need, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG  # workspace not 256-byte aligned
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_shared_expert_forward(16, 4, 256, 128, 16, 16, 16, 16, 16, 16, 16, 16, -1.0, 10.0, 256,
                                            need, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG  # limits must be positive


def test_routed_calibration_checks_arguments_on_host(binding):
    # ids / weights required (T > 0), sizes and top_k as the logit calibration
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_moe_calibrate_routed(16, None, 16, 0, 4, 256, 128, 4, 2, 16, 16, 16, 10.0, 10.0, 256,
                                           1 << 30, 16, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_moe_calibrate_routed(16, 16, 16, 0, 4, 256, 100, 4, 2, 16, 16, 16, 10.0, 10.0, 256,
                                           1 << 30, 16, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_UNSUPPORTED  # I % 128
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_moe_calibrate_routed(16, 16, 16, 0, 4, 256, 128, 2, 3, 16, 16, 16, 10.0, 10.0, 256,
                                           1 << 30, 16, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG and "top_k" in str(ei.value)
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_moe_calibrate_routed(16, 16, 16, 0, 4, 256, 128, 4, 2, 16, 16, 16, 10.0, 10.0, 256,
                                           1 << 30, None, 16, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG  # outputs required


def test_status_reader_and_debug_stall_check_arguments_on_host(binding):
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_read_device_status(None, stream=0)
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG
    with pytest.raises(binding.Nvfp4Error) as ei:
        binding.nvfp4_read_device_status(16, stream=0)  # not 256-byte aligned
    assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG
    for bad in (-1, 10001):
        with pytest.raises(binding.Nvfp4Error) as ei:
            binding.nvfp4_moe_set_debug_stall(bad)
        assert ei.value.status == binding.NVFP4_ERR_INVALID_ARG
    binding.nvfp4_moe_set_debug_stall(0)


def test_swap_l2_switch(binding):
    prev = binding.nvfp4_moe_set_swap_l2(1)
    try:
        assert prev == 0
        assert binding.nvfp4_moe_set_swap_l2(0) == 1
        with pytest.raises(binding.Nvfp4Error):
            binding.nvfp4_moe_set_swap_l2(2)
        assert binding.nvfp4_moe_set_swap_l2(0) == 0
    finally:
        binding.nvfp4_moe_set_swap_l2(prev)


def test_overlap_switch(binding):
    prev = binding.nvfp4_moe_set_overlap(0)
    try:
        assert prev == 1
        assert binding.nvfp4_moe_set_overlap(1) == 0
        with pytest.raises(binding.Nvfp4Error):
            binding.nvfp4_moe_set_overlap(2)
    finally:
        binding.nvfp4_moe_set_overlap(prev)
