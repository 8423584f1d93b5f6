"""The GEMM pipelines' bounded waits give up cleanly.

A plan created with W4A16_MOE_WAIT_TIMEOUT_NS set to 1 ns makes every
pipeline wait that has to wait at all give up at the next tick of the GPU
timer: the kernel raises its abort flag, drains the copies and MMAs it has in
flight (those drains keep the 2 s limit), frees its tensor memory and returns.
The forward's output is then meaningless, but nothing traps or hangs:
w4a16_moe_check_device_error reports W4A16_ERR_DEVICE_TIMEOUT, and the same
process runs a normal forward correctly afterwards.
"""
import pytest
import torch

from weight_only_int4_histogram_gb300 import _lib
from workloads import gen
from moe_testlib import case_on_gpu, compare, make_moe, oracle_rows, small_cfg

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from weight_only_int4_histogram_gb300 import build
    build.build()


@pytest.mark.parametrize("path", [1, 2], ids=["tc", "cc"])
def test_short_wait_limit_reports_timeout_and_context_survives(monkeypatch, path):
    # long K (28 pipeline stages per unit): the epilogue and dequant warps
    # certainly wait longer than one timer tick
    cfg = small_cfg(E=4, H=7168, I=256, k=2)
    T = 48
    w, x, ids, tw = case_on_gpu(cfg, T)
    monkeypatch.setenv("W4A16_MOE_WAIT_TIMEOUT_NS", "1")
    short = make_moe(cfg, T)
    monkeypatch.delenv("W4A16_MOE_WAIT_TIMEOUT_NS")
    short.set_gemm_path(path)
    short(x, w, tw, ids)
    torch.cuda.synchronize()
    with pytest.raises(_lib.W4A16Error) as ei:
        short.check_device_error()
    assert ei.value.status == 5  # W4A16_ERR_DEVICE_TIMEOUT
    # the flag was cleared by the read
    short.check_device_error()
    # the context is still usable: a plan with the default limit computes the right thing
    normal = make_moe(cfg, T)
    normal.set_gemm_path(path)
    out = normal(x, w, tw, ids)
    torch.cuda.synchronize()
    normal.check_device_error()
    compare(out, oracle_rows(cfg, w, x, ids, tw), "after a timed-out forward")


def test_short_wait_limit_with_fused_finalize(monkeypatch):
    # the fused CUDA-core launch with its finalize warp: every one of its waits
    # (stage, queue-space, record and ready waits) gives up cleanly too
    cfg = small_cfg(E=4, H=7168, I=256, k=2)
    T = 48
    w, x, ids, tw = case_on_gpu(cfg, T)
    monkeypatch.setenv("W4A16_MOE_WAIT_TIMEOUT_NS", "1")
    short = make_moe(cfg, T)
    monkeypatch.delenv("W4A16_MOE_WAIT_TIMEOUT_NS")
    short.set_gemm_path(2)
    short.set_fused_finalize(True)
    assert short.route_info(T).fused_finalize == 1
    short(x, w, tw, ids)
    torch.cuda.synchronize()
    with pytest.raises(_lib.W4A16Error) as ei:
        short.check_device_error()
    assert ei.value.status == 5  # W4A16_ERR_DEVICE_TIMEOUT
    normal = make_moe(cfg, T)
    normal.set_gemm_path(2)
    normal.set_fused_finalize(True)
    out = normal(x, w, tw, ids)
    torch.cuda.synchronize()
    normal.check_device_error()
    compare(out, oracle_rows(cfg, w, x, ids, tw), "fused finalize after a timed-out forward")


def test_short_wait_limit_one_group_fused_launch(monkeypatch):
    # the fused CUDA-core launch in its one-group form (two CTAs per SM, one
    # activation warp taking every stage): its waits give up cleanly as well
    cfg = small_cfg(E=4, H=7168, I=256, k=2)
    T = 48
    w, x, ids, tw = case_on_gpu(cfg, T)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    monkeypatch.setenv("W4A16_MOE_FUSED_GROUPS", "1")
    monkeypatch.setenv("W4A16_MOE_WAIT_TIMEOUT_NS", "1")
    short = make_moe(cfg, T)
    monkeypatch.delenv("W4A16_MOE_WAIT_TIMEOUT_NS")
    short.set_gemm_path(2)
    assert short.route_info(T).gemm1_ctas == 2 * sms
    short(x, w, tw, ids)
    torch.cuda.synchronize()
    with pytest.raises(_lib.W4A16Error) as ei:
        short.check_device_error()
    assert ei.value.status == 5  # W4A16_ERR_DEVICE_TIMEOUT
    normal = make_moe(cfg, T)
    normal.set_gemm_path(2)
    assert normal.route_info(T).gemm1_ctas == 2 * sms
    out = normal(x, w, tw, ids)
    torch.cuda.synchronize()
    normal.check_device_error()
    compare(out, oracle_rows(cfg, w, x, ids, tw), "one-group fused launch after a timed-out forward")
