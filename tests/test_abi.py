"""C-ABI checks that need no GPU: the library builds, loads and exports every
entry point include/w4a16_moe.h declares; descriptor validation and argument
checks return the documented status codes before any launch."""
import ctypes
import os
import re

import pytest

from weight_only_int4_histogram_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16_moe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_moe_\w+)\s*\(", src)))


def test_header_declares_the_binding_list():
    assert header_functions() == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert getattr(lib, name) is not None


def good_desc(**kw):
    d = dict(num_experts=8, expert_offset=0, hidden=256, inter=384, top_k=2, max_tokens=64,
             act=0, scale_kind=0, act_dtype=0)
    d.update(kw)
    return _lib.Desc(**d)


def test_plan_ok_and_workspace_positive(lib):
    plan, ws = _lib.w4a16_moe_plan(good_desc())
    assert ws > 0
    info = _lib.w4a16_moe_route_info(plan, 16)
    if info.gemm_path == _lib.PATH_TENSOR_CORES:
        assert info.tile_rows % 16 == 0 and 16 <= info.tile_rows <= 128
    else:
        assert info.tile_rows in (8, 16, 32)
    assert info.pipeline_stages >= 2
    _lib.w4a16_moe_plan_destroy(plan)


@pytest.mark.parametrize("kw,status", [
    (dict(num_experts=0), 2), (dict(num_experts=2000), 2), (dict(expert_offset=-1), 1),
    (dict(hidden=100), 2), (dict(inter=80), 2), (dict(hidden=48), 2), (dict(top_k=0), 2), (dict(top_k=17), 2),
    (dict(max_tokens=0), 2), (dict(act=5), 1), (dict(scale_kind=3), 1), (dict(act_dtype=2), 1),
])
def test_plan_rejects_bad_descriptors(lib, kw, status):
    with pytest.raises(_lib.W4A16Error) as ei:
        _lib.w4a16_moe_plan(good_desc(**kw))
    assert ei.value.status == status
    assert lib.w4a16_moe_last_error().decode() != ""


def test_calls_reject_bad_arguments_without_launching(lib):
    plan, ws = _lib.w4a16_moe_plan(good_desc())
    fake = 0x10000  # never dereferenced: validation fails first
    # T outside [0, max_tokens]
    with pytest.raises(_lib.W4A16Error) as ei:
        _lib.w4a16_moe_prepare_routes(plan, 65, fake, fake, 0)
    assert ei.value.status == 1
    # null ids
    with pytest.raises(_lib.W4A16Error):
        _lib.w4a16_moe_prepare_routes(plan, 4, 0, fake, 0)
    # misaligned workspace
    with pytest.raises(_lib.W4A16Error) as ei:
        _lib.w4a16_moe_prepare_routes(plan, 4, fake, fake + 8, 0)
    assert "aligned" in str(ei.value)
    # misaligned x in forward
    with pytest.raises(_lib.W4A16Error) as ei:
        _lib.w4a16_moe_forward(plan, 4, fake + 2, fake, fake, fake, fake, fake, fake, 0, fake, fake, 0)
    assert "x" in str(ei.value)
    # T = 0 is a no-op that succeeds even with null pointers
    _lib.w4a16_moe_prepare_routes(plan, 0, 0, 0, 0)
    _lib.w4a16_moe_forward(plan, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0)
    _lib.w4a16_moe_plan_destroy(plan)


def test_route_topk_rejects_bad_arguments_without_launching(lib):
    fake = 0x10000  # never dereferenced: validation fails first
    for args, status in [((fake, -1, 8, 2, fake, fake), 1),       # negative num_tokens
                         ((fake, 4, 0, 1, fake, fake), 2),        # num_global < 1
                         ((fake, 4, 1025, 8, fake, fake), 2),     # num_global > 1024
                         ((fake, 4, 8, 0, fake, fake), 2),        # top_k < 1
                         ((fake, 4, 8, 9, fake, fake), 2),        # top_k > num_global
                         ((fake, 4, 64, 17, fake, fake), 2),      # top_k > 16
                         ((0, 4, 8, 2, fake, fake), 1),           # null logits
                         ((fake + 2, 4, 8, 2, fake, fake), 1),    # misaligned logits
                         ((fake, 4, 8, 2, fake, 0), 1)]:          # null weights
        with pytest.raises(_lib.W4A16Error) as ei:
            _lib.w4a16_moe_route_topk(*args, 0)
        assert ei.value.status == status, args
    # an empty batch succeeds even with null pointers
    _lib.w4a16_moe_route_topk(0, 0, 8, 2, 0, 0, 0)


def test_forward_masked_validates_plan_and_sizes(lib):
    fake = 0x10000  # never dereferenced: validation fails first
    plan8, _ = _lib.w4a16_moe_plan(good_desc())  # top_k 2
    with pytest.raises(_lib.W4A16Error) as ei:
        _lib.w4a16_moe_forward_masked(plan8, 4, fake, fake, fake, fake, fake, fake, fake, fake, 0)
    assert ei.value.status == 2 and "top_k" in str(ei.value)
    _lib.w4a16_moe_plan_destroy(plan8)
    plan1, _ = _lib.w4a16_moe_plan(good_desc(top_k=1, max_tokens=64))
    E = good_desc().num_experts
    with pytest.raises(_lib.W4A16Error) as ei:  # more rows than max_tokens
        _lib.w4a16_moe_forward_masked(plan1, 64 // E + 1, fake, fake, fake, fake, fake, fake, fake, fake, 0)
    assert ei.value.status == 1
    with pytest.raises(_lib.W4A16Error):  # negative max_rows
        _lib.w4a16_moe_forward_masked(plan1, -1, fake, fake, fake, fake, fake, fake, fake, fake, 0)
    with pytest.raises(_lib.W4A16Error):  # null counts
        _lib.w4a16_moe_forward_masked(plan1, 2, 0, fake, fake, fake, fake, fake, fake, fake, 0)
    _lib.w4a16_moe_forward_masked(plan1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0)  # no rows: no-op
    _lib.w4a16_moe_plan_destroy(plan1)


def test_overrides_validate_and_resize_workspace(lib):
    plan, ws = _lib.w4a16_moe_plan(good_desc())
    with pytest.raises(_lib.W4A16Error):
        _lib.w4a16_moe_set_overrides(plan, 24, 0, 0)
    with pytest.raises(_lib.W4A16Error):
        _lib.w4a16_moe_set_overrides(plan, 0, 65, 0)
    _lib.w4a16_moe_set_gemm_path(plan, _lib.PATH_TENSOR_CORES)  # tile_rows applies to this path
    ws2 = _lib.w4a16_moe_set_overrides(plan, 128, 4, 2)
    info = _lib.w4a16_moe_route_info(plan, 16)
    assert info.tile_rows == 128 and info.gemm1_splits == 4 and info.gemm2_splits == 2
    assert ws2 >= ws
    _lib.w4a16_moe_set_overrides(plan, 0, 0, 0)
    _lib.w4a16_moe_plan_destroy(plan)


def test_planner_tile_height_follows_route_counts(lib):
    """Route-count-based tile selection: taller route tiles as routes per
    expert grow (LMDeploy page, Modification)."""
    plan, _ = _lib.w4a16_moe_plan(good_desc(num_experts=384, hidden=7168, inter=256, top_k=8,
                                            max_tokens=2048))
    bns = [_lib.w4a16_moe_route_info(plan, t).tile_rows for t in (1, 8, 32, 256, 1024, 2048)]
    # CUDA-core GEMV tiles (8 routes) for the smallest batches, then tensor-core tiles
    assert bns == sorted(bns) and bns[0] == 8 and bns[-1] >= 64
    s1 = [_lib.w4a16_moe_route_info(plan, t).gemm1_splits for t in (1, 2048)]
    assert s1[0] > 1 and s1[1] == 1  # split-K only for small batches
    _lib.w4a16_moe_plan_destroy(plan)


def test_global_experts_set_the_routing_density(lib):
    """A declared global expert count makes the planner expect T * k / global
    routes per local expert (an expert-parallel shard's share), not T * k / E:
    32 local of 256 global experts, H 7168, I 2048, top-8 -> 2 routes per local
    expert at 64 tokens: CUDA cores with 8-route tiles; undeclared, the same
    shard is planned for 16 routes per expert.  Results never depend on it;
    fewer global than local experts is refused."""
    shard = dict(num_experts=32, expert_offset=64, hidden=7168, inter=2048, top_k=8, max_tokens=4096)
    plan, _ = _lib.w4a16_moe_plan(good_desc(global_experts=256, **shard))
    info = _lib.w4a16_moe_route_info(plan, 64)
    assert info.gemm_path == _lib.PATH_CUDA_CORES and info.tile_rows == 8
    # 11 routes per local expert at 352 tokens; tensor cores above
    assert _lib.w4a16_moe_route_info(plan, 352).gemm_path == _lib.PATH_CUDA_CORES
    assert _lib.w4a16_moe_route_info(plan, 353).gemm_path == _lib.PATH_TENSOR_CORES
    _lib.w4a16_moe_plan_destroy(plan)
    plan, _ = _lib.w4a16_moe_plan(good_desc(**shard))
    assert _lib.w4a16_moe_route_info(plan, 64).tile_rows == 32
    _lib.w4a16_moe_plan_destroy(plan)
    with pytest.raises(_lib.W4A16Error) as ei:
        _lib.w4a16_moe_plan(good_desc(global_experts=16, **shard))
    assert ei.value.status == 1


def test_fused_launch_compute_groups(lib, monkeypatch):
    """The fused CUDA-core launch: one compute group per CTA and two CTAs per SM
    (grid 2 x SMs, a ring of 4 stages at 8-route tiles, 3 at 16) once the
    expected gate/up units fill 1.9 waves of those CTAs -- on the Kimi shard
    from 24 tokens (1.99 waves), not at 16 (1.43) -- else two groups per CTA and
    one CTA per SM.  Never with the fused finalize; W4A16_MOE_FUSED_GROUPS
    forces either form."""
    desc = good_desc(num_experts=384, hidden=7168, inter=256, top_k=8, max_tokens=2048)
    plan, _ = _lib.w4a16_moe_plan(desc)
    sms = _lib.w4a16_moe_route_info(plan, 1).gemm1_ctas  # one CTA per SM at one token
    info = {t: _lib.w4a16_moe_route_info(plan, t) for t in (1, 8, 16, 24, 32, 64, 256)}
    assert all(i.fused_gemms == 1 for i in info.values())
    assert {t: i.gemm1_ctas // sms for t, i in info.items()} == {1: 1, 8: 1, 16: 1, 24: 2, 32: 2, 64: 2, 256: 2}
    assert info[32].tile_rows == 8 and info[32].pipeline_stages == 4 and info[32].gemm2_ctas == 2 * sms
    assert info[256].tile_rows == 16 and info[256].pipeline_stages == 3
    _lib.w4a16_moe_set_fused_finalize(plan, True)
    assert _lib.w4a16_moe_route_info(plan, 32).gemm1_ctas == sms
    _lib.w4a16_moe_plan_destroy(plan)
    monkeypatch.setenv("W4A16_MOE_FUSED_GROUPS", "2")
    plan, _ = _lib.w4a16_moe_plan(desc)
    assert _lib.w4a16_moe_route_info(plan, 32).gemm1_ctas == sms
    _lib.w4a16_moe_plan_destroy(plan)
    monkeypatch.setenv("W4A16_MOE_FUSED_GROUPS", "1")
    plan, _ = _lib.w4a16_moe_plan(desc)
    assert _lib.w4a16_moe_route_info(plan, 16).gemm1_ctas == 2 * sms
    _lib.w4a16_moe_plan_destroy(plan)


def test_gemm_path_choice_and_validation(lib):
    """Few routes per expert -> CUDA-core GEMV with 8- to 32-route tiles; many ->
    tensor cores (above 11 routes per expert with group scales, 24 with
    per-channel scales); forced paths hold at every batch size."""
    plan, _ = _lib.w4a16_moe_plan(good_desc(num_experts=384, hidden=7168, inter=256, top_k=8,
                                            max_tokens=2048))
    # 384 experts, top-8, group scales: 11 routes per expert at 528 tokens
    paths = {t: _lib.w4a16_moe_route_info(plan, t).gemm_path for t in (1, 32, 528, 529, 2048)}
    assert paths == {1: _lib.PATH_CUDA_CORES, 32: _lib.PATH_CUDA_CORES, 528: _lib.PATH_CUDA_CORES,
                     529: _lib.PATH_TENSOR_CORES, 2048: _lib.PATH_TENSOR_CORES}
    assert _lib.w4a16_moe_route_info(plan, 32).tile_rows == 8
    with pytest.raises(_lib.W4A16Error) as ei:
        _lib.w4a16_moe_set_gemm_path(plan, 3)
    assert ei.value.status == 1
    ws_cc = _lib.w4a16_moe_set_gemm_path(plan, _lib.PATH_CUDA_CORES)
    info = _lib.w4a16_moe_route_info(plan, 2048)
    assert info.gemm_path == _lib.PATH_CUDA_CORES and info.tile_rows == 32
    # tile_rows overrides apply to the tensor-core path only
    _lib.w4a16_moe_set_overrides(plan, 64, 0, 0)
    assert _lib.w4a16_moe_route_info(plan, 2048).tile_rows == 32
    _lib.w4a16_moe_set_gemm_path(plan, _lib.PATH_TENSOR_CORES)
    assert _lib.w4a16_moe_route_info(plan, 1).gemm_path == _lib.PATH_TENSOR_CORES
    assert _lib.w4a16_moe_route_info(plan, 1).tile_rows == 64
    _lib.w4a16_moe_set_overrides(plan, 0, 0, 0)
    ws_auto = _lib.w4a16_moe_set_gemm_path(plan, _lib.PATH_AUTO)
    assert ws_cc > 0 and ws_auto > 0
    _lib.w4a16_moe_plan_destroy(plan)
    # per-channel scales (scale_kind 1): 24 routes per expert, E 60 top-4 -> 360 tokens
    plan, _ = _lib.w4a16_moe_plan(good_desc(num_experts=60, hidden=2048, inter=1408, top_k=4,
                                            scale_kind=1, max_tokens=1024))
    paths = {t: _lib.w4a16_moe_route_info(plan, t).gemm_path for t in (8, 360, 361, 1024)}
    assert paths == {8: _lib.PATH_CUDA_CORES, 360: _lib.PATH_CUDA_CORES, 361: _lib.PATH_TENSOR_CORES,
                     1024: _lib.PATH_TENSOR_CORES}
    _lib.w4a16_moe_plan_destroy(plan)
