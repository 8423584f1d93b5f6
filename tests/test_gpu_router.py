"""GPU parity of the router step (softmax + top-k, ``w4a16_moe_route_topk``)
against the CPU oracle, and the route-prep/forward chain fed by it.

Expert ids are compared bit for bit (both sides order the FP32 logits
exactly, ties to the lower index); weights are FP32 softmax probabilities
against the oracle's double ones, relative tolerance 1e-5 (a handful of FP32
roundings in exp, the sum and the division)."""
import numpy as np
import pytest
import torch

import oracle
from workloads import gen
from moe_testlib import compare, make_moe, oracle_rows, small_cfg

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import weight_only_int4_histogram_gb300 as W  # noqa: E402


def check(logits, k):
    ids, w = W.route_topk(logits, k)
    torch.cuda.synchronize()
    want_ids, want_w = oracle.route_topk(logits.cpu(), k)
    np.testing.assert_array_equal(ids.cpu().numpy(), want_ids)
    np.testing.assert_allclose(w.cpu().numpy().astype(np.float64), want_w, rtol=1e-5, atol=1e-12)


@pytest.mark.parametrize("name", list(gen.CONFIGS))
def test_workload_logits(name):
    cfg = gen.CONFIGS[name]
    for T in (1, 7, 256, 2048):
        check(gen.make_logits(cfg, T, "cuda"), cfg.top_k)


@pytest.mark.parametrize("G,k", [(1, 1), (5, 5), (31, 3), (33, 16), (64, 6), (1000, 7), (1024, 16)])
def test_shapes_and_ragged_lanes(G, k):
    g = torch.Generator(device="cuda").manual_seed(G * 100 + k)
    check(torch.randn(37, G, generator=g, device="cuda"), k)


def test_ties_take_the_lower_index():
    G, k = 96, 8
    lg = torch.zeros(4, G, device="cuda")
    lg[1, 40:48] = 1.0  # eight equal winners
    lg[2, :] = torch.arange(G, device="cuda").float().remainder(3)  # many ties at 2.0
    lg[3, 90] = 5.0
    check(lg, k)
    ids, _ = W.route_topk(lg, k)
    assert ids[0].tolist() == list(range(8))
    assert ids[1].tolist() == list(range(40, 48))


def test_empty_batch_is_a_no_op():
    ids, w = W.route_topk(torch.zeros(0, 16, device="cuda"), 4)
    assert ids.shape == (0, 4) and w.shape == (0, 4)


def test_router_then_forward_matches_generator_routes():
    """route_topk -> prepare_routes -> forward on a local shard of 16 of 64
    experts (ids of other ranks are masked by the plan's expert range) equals
    the oracle on the same routes, and the routes equal the input generator's
    (torch softmax + top-k of the same logits)."""
    cfg = small_cfg(E=16, H=512, I=256, k=4, seed=31, global_experts=64, expert_offset=16)
    T = 40
    w = gen.make_weights(cfg, "cuda")
    x = gen.make_activations(cfg, T, "cuda")
    logits = gen.make_logits(cfg, T, "cuda")
    ids, tw = W.route_topk(logits, cfg.top_k)
    gen_ids, gen_w = gen.make_routes(cfg, T, "cuda")
    local = (ids >= cfg.expert_offset) & (ids < cfg.expert_offset + cfg.num_experts)
    assert torch.equal(torch.where(local, ids, torch.full_like(ids, -1)), gen_ids)
    torch.testing.assert_close(tw, gen_w, rtol=1e-5, atol=1e-7)
    moe = make_moe(cfg, T)
    out = moe(x, w, tw, ids)
    torch.cuda.synchronize()
    compare(out, oracle_rows(cfg, w, x, ids, tw), "router -> forward")


@pytest.mark.parametrize("name,T", [("kimi_tp8_e384_h7168_i256_k8", 1), ("kimi_tp8_e384_h7168_i256_k8", 33),
                                    ("kimi_tp8_e384_h7168_i256_k8", 2048),
                                    ("deepseek_local_e32of256_h7168_i2048_k8", 512),
                                    ("relu2_skew_e64_h2688_i1856_k6", 4096), ("tiny_e8_h256_i384_k2", 16)])
def test_route_and_prepare_matches_router_then_prepare(name, T):
    """The fused router + route preparation gives the router's ids and
    weights bit for bit and the oracle's route layout bit for bit."""
    cfg = gen.CONFIGS[name]
    logits = gen.make_logits(cfg, T, "cuda")
    moe = make_moe(cfg, T)
    ids, w = moe.route_and_prepare(logits)
    torch.cuda.synchronize()
    rid, rw = W.route_topk(logits, cfg.top_k)
    torch.cuda.synchronize()
    assert torch.equal(ids, rid)
    assert torch.equal(w.view(torch.int32), rw.view(torch.int32))
    got = moe.read_route_layout(T)
    want = oracle.prepare_routes(cfg, ids.cpu(), got["tile_rows"])
    for key in ("counts", "offs", "perm", "inv", "tiles"):
        np.testing.assert_array_equal(got[key].numpy(), want[key], err_msg=key)


def test_route_and_prepare_then_forward():
    cfg = small_cfg(E=16, H=512, I=256, k=4, expert_offset=16)
    T = 70
    w = gen.make_weights(cfg, "cuda")
    x = gen.make_activations(cfg, T, "cuda")
    logits = torch.randn(T, 64, device="cuda", generator=torch.Generator(device="cuda").manual_seed(7))
    moe = make_moe(cfg, T)
    ids, tw = moe.route_and_prepare(logits)
    out = moe.forward(x, w, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    compare(out, oracle_rows(cfg, w, x, ids, tw), "route_and_prepare + forward")
