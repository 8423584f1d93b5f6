"""GPU checks of the fused CUDA-core launch (both expert GEMMs fed from one
device work queue) and of the deterministic fused finalize.

* fused forwards match the oracle within the parity tolerance, on every
  activation / scale / dtype / layout combination, with invalid and masked
  routes, at token counts that give split gate/up units and mixed route-block
  heights;
* the fused finalize (combine inside the down epilogue, no data atomics) is
  bit-identical to the separate combine launch, renormalised or not, with
  tokens that have no valid route (exact zero rows);
* forwards are bit-identical when repeated, and a forward that reuses a route
  layout (no prepare_routes in between) is still correct: the queue state is
  reset by the combine, or by the last CTA when the finalize is fused;
* the fused and the two-launch CUDA-core forwards agree within tolerance;
* the one-group form of the fused launch (one compute group per CTA, two CTAs
  per SM, 8-route tiles) matches the oracle on every combination, repeats bit
  for bit and agrees with the two-group form; the planner takes it on the
  Kimi shard at 32 tokens.
"""
import numpy as np
import pytest
import torch

from workloads import gen
from moe_testlib import case_on_gpu, compare, make_moe, oracle_rows, small_cfg

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

CC = 2  # W4A16_PATH_CUDA_CORES

SHAPES = [
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_FP16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_FP16),
]


@pytest.fixture(scope="module", autouse=True)
def _build():
    from weight_only_int4_histogram_gb300 import build
    build.build()


def fused_moe(cfg, T, finalize=False, interleaved=False, w=None):
    moe = make_moe(cfg, T)
    moe.set_gemm_path(CC)
    moe.set_fused_finalize(finalize)
    info = moe.route_info(T)
    assert info.fused_gemms == 1 and info.fused_finalize == int(finalize)
    wl = moe.relayout_weights(w) if interleaved else w
    return moe, wl


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"a{s['act']}s{s['scale']}d{s['dt']}")
@pytest.mark.parametrize("T", [1, 3, 17, 40])
@pytest.mark.parametrize("interleaved", [False, True], ids=["ckpt", "il"])
def test_fused_matches_oracle_and_finalize_is_bit_identical(shape, T, interleaved):
    # H = 1056: 5 gate/up K blocks (ragged last), I = 320: a half-used SwiGLU
    # tile and 2-stage down units; E = 7 experts with k = 3 over 1..40 tokens
    # gives split gate/up units (small T) and mixed route-block heights
    cfg = small_cfg(E=7, H=1056, I=320, k=3, **shape)
    w, x, ids, tw = case_on_gpu(cfg, T)
    base, wl = fused_moe(cfg, T, finalize=False, interleaved=interleaved, w=w)
    want = base(x, wl, tw, ids).clone()
    torch.cuda.synchronize()
    base.check_device_error()
    compare(want, oracle_rows(cfg, w, x, ids, tw), f"fused {cfg.name} T={T}")
    fin, wl2 = fused_moe(cfg, T, finalize=True, interleaved=interleaved, w=w)
    got = fin(x, wl2, tw, ids)
    torch.cuda.synchronize()
    fin.check_device_error()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("finalize", [False, True], ids=["combine", "finalize"])
def test_invalid_routes_renormalize_and_empty_tokens(finalize):
    cfg = small_cfg(E=8, H=768, I=256, k=4, global_experts=32, expert_offset=8)
    T = 23
    w, x, ids, tw = case_on_gpu(cfg, T)
    ids = ids.clone()
    # ids are global: local experts are 8..15; mask some routes, push some out
    # of range, and leave tokens 5 and 11 without any valid route
    ids[::3, 0] = -1
    ids[1::4, 1] = 31
    ids[5, :] = -1
    ids[11, :] = 2
    moe, _ = fused_moe(cfg, T, finalize=finalize, w=w)
    for renorm in (False, True):
        out = torch.full((T, cfg.hidden), float("nan"), dtype=cfg.torch_act_dtype(), device="cuda")
        moe(x, w, tw, ids, renormalize=renorm, out=out)
        torch.cuda.synchronize()
        moe.check_device_error()
        assert torch.all(out[5].view(torch.int16) == 0) and torch.all(out[11].view(torch.int16) == 0)
        compare(out, oracle_rows(cfg, w, x, ids, tw, renormalize=renorm), f"fin={finalize} renorm={renorm}")
        ref, _ = fused_moe(cfg, T, finalize=not finalize, w=w)
        other = ref(x, w, tw, ids, renormalize=renorm)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), other.view(torch.int16))


@pytest.mark.parametrize("finalize", [False, True], ids=["combine", "finalize"])
def test_reused_route_layout_and_repeat_bit_identical(finalize):
    cfg = small_cfg(E=16, H=1024, I=512, k=4, seed=31)
    T = 9
    w, x, ids, tw = case_on_gpu(cfg, T)
    moe, _ = fused_moe(cfg, T, finalize=finalize, w=w)
    first = moe(x, w, tw, ids).clone()
    # two more forwards on the same route layout (no prepare_routes between),
    # with other activations: each must be right, not a stale result
    for i in range(2):
        x2 = gen.make_activations(cfg, T, "cuda", seed=500 + i)
        out = moe.forward(x2, w, tw, ids)
        torch.cuda.synchronize()
        moe.check_device_error()
        compare(out, oracle_rows(cfg, w, x2, ids, tw), f"reuse {i} fin={finalize}")
    again = moe(x, w, tw, ids)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), first.view(torch.int16))


def test_fused_and_two_launch_paths_agree(monkeypatch):
    cfg = small_cfg(E=12, H=2048, I=512, k=4, seed=41)
    for T in (2, 12, 33):
        w, x, ids, tw = case_on_gpu(cfg, T)
        monkeypatch.setenv("W4A16_MOE_FUSED", "0")
        two = make_moe(cfg, T)
        monkeypatch.delenv("W4A16_MOE_FUSED")
        two.set_gemm_path(CC)
        assert two.route_info(T).fused_gemms == 0
        a = two(x, w, tw, ids).clone()
        one, _ = fused_moe(cfg, T, w=w)
        b = one(x, w, tw, ids)
        torch.cuda.synchronize()
        ref = oracle_rows(cfg, w, x, ids, tw)
        compare(a, ref, f"two launches T={T}")
        compare(b, ref, f"fused T={T}")


@pytest.mark.parametrize("T", [1, 8, 32])
def test_full_size_kimi_fused_finalize_sampled_rows(monkeypatch, T):
    cfg = gen.CONFIGS["kimi_tp8_e384_h7168_i256_k8"]
    w = gen.make_weights(cfg, "cuda")
    _, x, ids, tw = case_on_gpu(cfg, T, weights_gpu=w)
    # the finalize runs with two compute groups per CTA: the combine-launch
    # forward it must equal bit for bit sums each unit the same way
    monkeypatch.setenv("W4A16_MOE_FUSED_GROUPS", "2")
    base, wl = fused_moe(cfg, T, finalize=False, interleaved=True, w=w)
    want = base(x, wl, tw, ids).clone()
    fin, wl2 = fused_moe(cfg, T, finalize=True, interleaved=True, w=w)
    got = fin(x, wl2, tw, ids)
    torch.cuda.synchronize()
    fin.check_device_error()
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    rows = sorted(set([0, T - 1] + np.random.default_rng(T).integers(0, T, size=min(T, 12)).tolist()))
    compare(got[rows], oracle_rows(cfg, w, x, ids, tw, rows=rows), f"kimi T={T} fused finalize")


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"a{s['act']}s{s['scale']}d{s['dt']}")
@pytest.mark.parametrize("interleaved", [False, True], ids=["ckpt", "il"])
def test_one_compute_group_per_cta(monkeypatch, shape, interleaved):
    # 64 experts, k = 2 over 40 tokens: 1.25 routes per expert (8-route tiles);
    # H = 1056: 5 gate/up K blocks (ragged last) that one group walks alone
    cfg = small_cfg(E=64, H=1056, I=320, k=2, seed=53, **shape)
    T = 40
    w, x, ids, tw = case_on_gpu(cfg, T)
    outs = {}
    for groups in ("1", "2"):
        monkeypatch.setenv("W4A16_MOE_FUSED_GROUPS", groups)
        moe, wl = fused_moe(cfg, T, interleaved=interleaved, w=w)
        info = moe.route_info(T)
        assert info.tile_rows == 8
        assert info.gemm1_ctas == (2 if groups == "1" else 1) * _sms()
        out = moe(x, wl, tw, ids).clone()
        again = moe(x, wl, tw, ids)
        torch.cuda.synchronize()
        moe.check_device_error()
        assert torch.equal(again.view(torch.int16), out.view(torch.int16))
        outs[groups] = out
    ref = oracle_rows(cfg, w, x, ids, tw)
    compare(outs["1"], ref, f"one group {cfg.name}")
    compare(outs["2"], ref, f"two groups {cfg.name}")
    compare(outs["1"], outs["2"].float().cpu().numpy(), f"one vs two groups {cfg.name}")


def test_full_size_kimi_one_group_sampled_rows():
    """The planner's choice at 32 tokens on the Kimi shard: one compute group
    per CTA, two CTAs per SM."""
    cfg = gen.CONFIGS["kimi_tp8_e384_h7168_i256_k8"]
    T = 32
    w = gen.make_weights(cfg, "cuda")
    _, x, ids, tw = case_on_gpu(cfg, T, weights_gpu=w)
    moe, wl = fused_moe(cfg, T, interleaved=True, w=w)
    assert moe.route_info(T).gemm1_ctas == 2 * _sms()
    out = moe(x, wl, tw, ids).clone()
    again = moe(x, wl, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))
    rows = sorted(set([0, T - 1] + np.random.default_rng(7).integers(0, T, size=10).tolist()))
    compare(out[rows], oracle_rows(cfg, w, x, ids, tw, rows=rows), "kimi T=32 one group")
