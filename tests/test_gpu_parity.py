"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Sizes span several route tiles, weight tiles and K blocks with ragged tails;
full-size workloads are checked on sampled tokens in the launch configuration
the benchmark times.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import gen
from moe_testlib import compare, make_moe, case_on_gpu, oracle_rows, small_cfg

# GEMM paths: tensor cores (tcgen05) and the CUDA-core GEMV for few routes per expert
PATHS = {"tc": 1, "cc": 2}

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from weight_only_int4_histogram_gb300 import build
    build.build()


# ---------------------------------------------------------------------------
# route preparation: bit-exact
# ---------------------------------------------------------------------------

def check_routes(moe, cfg, ids):
    T = ids.shape[0]
    moe.prepare_routes(ids)
    torch.cuda.synchronize()
    got = moe.read_route_layout(T)
    want = oracle.prepare_routes(cfg, ids.cpu(), got["tile_rows"])
    np.testing.assert_array_equal(got["counts"].numpy(), want["counts"])
    np.testing.assert_array_equal(got["offs"].numpy(), want["offs"])
    np.testing.assert_array_equal(got["perm"].numpy(), want["perm"])
    np.testing.assert_array_equal(got["inv"].numpy(), want["inv"])
    assert got["num_tiles"] == want["num_tiles"]
    np.testing.assert_array_equal(got["tiles"].numpy(), want["tiles"])


@pytest.mark.parametrize("name", list(gen.CONFIGS))
def test_route_prep_bit_exact_on_workloads(name):
    cfg = gen.CONFIGS[name]
    moe = make_moe(cfg, max(cfg.tokens))
    for T in cfg.tokens:
        ids, _ = gen.make_routes(cfg, T, "cuda")
        check_routes(moe, cfg, ids)


@pytest.mark.parametrize("seed", range(8))
def test_route_prep_bit_exact_fuzz(seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.choice([1, 3, 8, 33, 384, 1024]))
    k = int(rng.choice([1, 2, 3, 4, 6, 8]))
    T = int(rng.integers(1, 700))
    off = int(rng.integers(0, 5))
    cfg = gen.MoEConfig("fuzz", E, 256, 256, k, expert_offset=off)
    moe = make_moe(cfg, 700)
    if seed % 4 == 1:
        moe.set_overrides(tile_rows=int(rng.choice([16, 32, 64, 128])))
    frac_invalid = [0.0, 0.3, 1.0, 0.05][seed % 4]
    ids = rng.integers(off, off + E, size=(T, k))
    ids = np.where(rng.random((T, k)) < frac_invalid, -1, ids)
    ids = np.where(rng.random((T, k)) < 0.05, off + E + 7, ids)  # masked (other rank)
    if seed == 5:
        ids[:] = off  # every route on one expert
    check_routes(moe, cfg, torch.from_numpy(ids.astype(np.int32)).cuda())


# ---------------------------------------------------------------------------
# MoE output parity
# ---------------------------------------------------------------------------

def run_and_compare(cfg, T, overrides=None, renormalize=False, ids=None, what="", path=None):
    w, x, ids_, tw = case_on_gpu(cfg, T)
    if ids is not None:
        ids_ = ids.cuda()
    moe = make_moe(cfg, max(T, 1))
    if path is not None:
        moe.set_gemm_path(PATHS[path])
        assert moe.route_info(T).gemm_path == PATHS[path]
    if overrides:
        moe.set_overrides(**overrides)
    out = moe(x, w, tw, ids_, renormalize=renormalize)
    torch.cuda.synchronize()
    moe.check_device_error()
    ref = oracle_rows(cfg, w, x, ids_, tw, renormalize=renormalize)
    return compare(out, ref, what or f"{cfg.name} T={T} {overrides} {path}"), (moe, w, x, ids_, tw, out)


def test_tiny_workload_parity():
    cfg = gen.TINY
    run_and_compare(cfg, 16)


SHAPES = [
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_FP16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_FP16),
]


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"a{s['act']}s{s['scale']}d{s['dt']}")
@pytest.mark.parametrize("T", [1, 7, 61])
def test_small_shapes_parity(shape, T, path):
    # H = 704: 2 full K blocks + a ragged one; I = 320: ragged weight tiles
    cfg = small_cfg(E=5, H=704, I=320, k=3, **shape)
    run_and_compare(cfg, T, path=path)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"a{s['act']}s{s['scale']}d{s['dt']}")
@pytest.mark.parametrize("relaid", [False, True], ids=["ckpt", "il"])
def test_sizes_that_are_odd_multiples_of_32(shape, path, relaid):
    """H = 1056 (33 groups of 32: group-scale rows of 66 bytes, only 2-byte
    aligned; a partial last 64-column activation box and 256-K stage) and
    I = 352 (a half-used last SwiGLU tile pair, a partial last stage of the
    down GEMM)."""
    cfg = small_cfg(E=5, H=1056, I=352, k=3, **shape)
    T = 29
    w, x, ids, tw = case_on_gpu(cfg, T)
    moe = make_moe(cfg, T)
    moe.set_gemm_path(PATHS[path])
    wts = moe.relayout_weights(w) if relaid else w
    out = moe(x, wts, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    compare(out, oracle_rows(cfg, w, x, ids, tw), f"{cfg.name} {path} relaid={relaid}")


@pytest.mark.parametrize("path", list(PATHS))
def test_cuda_graph_replay_at_k_1056(path):
    """"feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), Validation:
    full MoE CUDA-graph replay at K = 1056 -- here hidden 1056 (the gate/up
    GEMM's K) and inter 1056 (the down GEMM's K), new inputs copied into the
    captured buffers before each replay."""
    cfg = small_cfg(E=6, H=1056, I=1056, k=2, seed=13)
    T = 37
    w, x, ids, tw = case_on_gpu(cfg, T)
    moe = make_moe(cfg, T)
    moe.set_gemm_path(PATHS[path])
    out = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe(x, w, tw, ids, out=out, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe(x, w, tw, ids, out=out, stream=s)
    for trial in range(2):
        x2 = gen.make_activations(cfg, T, "cuda", seed=300 + trial)
        ids2, tw2 = gen.make_routes(cfg, T, "cuda", seed=400 + trial)
        x.copy_(x2)
        ids.copy_(ids2)
        tw.copy_(tw2)
        g.replay()
        torch.cuda.synchronize()
        moe.check_device_error()
        compare(out, oracle_rows(cfg, w, x2, ids2, tw2), f"K=1056 graph replay {trial} {path}")


def bucket_ids(E, counts, k, seed=0):
    """ids [T, k] giving expert e exactly counts[e] routes (remaining slots
    -1), tokens shuffled."""
    rng = np.random.default_rng(seed)
    flat = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    T = -(-len(flat) // k)
    flat = np.concatenate([flat, np.full(T * k - len(flat), -1)])
    rng.shuffle(flat)
    return torch.from_numpy(flat.reshape(T, k).astype(np.int32)), T


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"a{s['act']}s{s['scale']}d{s['dt']}")
def test_cuda_core_route_count_buckets(shape):
    """Experts with 1, 2, 3, 4, 5, 8, 9, 16, 17 and 40 routes: every route-count
    specialisation of the CUDA-core GEMV, full and partial 16-route tiles, and
    experts spanning several tiles."""
    counts = [1, 2, 3, 4, 5, 8, 9, 16, 17, 40, 0]
    cfg = small_cfg(E=len(counts), H=640, I=192, k=4, **shape)
    ids, T = bucket_ids(cfg.num_experts, counts, cfg.top_k)
    run_and_compare(cfg, T, ids=ids, path="cc")


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2], SHAPES[3]], ids=lambda s: f"s{s['scale']}d{s['dt']}")
@pytest.mark.parametrize("mag", ["tiny", "huge", "mixed"])
def test_activation_magnitudes(shape, mag, path):
    """Activations far from unit scale (the CUDA-core path rescales them by
    powers of two before its FP16 sums): per-token factors 2^-20 .. 2^12 for
    BF16, 2^-2 .. 2^3 for FP16 (outputs grow like the factor squared and would
    otherwise leave FP16's normal range in the final cast)."""
    cfg = small_cfg(E=4, H=512, I=256, k=2, **shape)
    T = 24
    lo, hi = (-20, 12) if shape["dt"] == gen.DT_BF16 else (-2, 3)
    if mag == "tiny":
        f = torch.full((T, 1), 2.0 ** lo)
    elif mag == "huge":
        f = torch.full((T, 1), 2.0 ** hi)
    else:
        f = 2.0 ** torch.linspace(lo, hi, T).round().reshape(T, 1)
    w, x, ids, tw = case_on_gpu(cfg, T)
    x = (x.float() * f.cuda()).to(x.dtype)
    moe = make_moe(cfg, T)
    moe.set_gemm_path(PATHS[path])
    out = moe(x, w, tw, ids)
    torch.cuda.synchronize()
    ref = oracle_rows(cfg, w, x, ids, tw)
    # each token's output scales with its factor: compare token by token
    for t in range(T):
        compare(out[t:t + 1], ref[t:t + 1], f"{mag} token {t} {path}")


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("scale", [gen.SCALE_GROUP32, gen.SCALE_PER_CHANNEL])
def test_fp16_outputs_in_the_subnormal_range(scale, path):
    """FP16 activations scaled by 2^-7: the expert outputs (quadratic in x
    through the gated MLP) land in FP16's subnormal range, where the final
    cast itself moves values by up to half of 2^-24.  The reference is then
    the oracle's own FP16 output (its FP32 accumulator cast once): both sides
    round the same FP32 sum to the same grid, so they are compared element by
    element, within the parity bars plus one subnormal step."""
    cfg = small_cfg(E=4, H=512, I=256, k=2, scale=scale, dt=gen.DT_FP16)
    T = 24
    w, x, ids, tw = case_on_gpu(cfg, T)
    x = (x.float() * 2.0 ** -7).to(x.dtype)
    moe = make_moe(cfg, T)
    moe.set_gemm_path(PATHS[path])
    out = moe(x, w, tw, ids)
    torch.cuda.synchronize()
    _, bits = oracle.moe_forward(cfg, x.cpu(), w.to("cpu"), tw.cpu(), ids.cpu())
    ref = oracle.fp16_decode(bits)
    g = out.float().cpu().numpy().astype(np.float64)
    assert (np.abs(ref[ref != 0]) < 2.0 ** -14).mean() > 0.5, "case must exercise subnormal outputs"
    step = 2.0 ** -24
    err = np.abs(g - ref)
    assert err.max() <= 2e-2 * np.abs(ref).max() + step, (err.max(), np.abs(ref).max())
    assert np.linalg.norm(g - ref) <= 5e-3 * np.linalg.norm(ref) + step * np.sqrt(ref.size)


@pytest.mark.parametrize("tile_rows", [16, 32, 48, 128])
def test_route_tile_heights(tile_rows):
    """Route-tile boundary cases: full tiles plus partial tails at several
    heights, top-k 2 and 3."""
    for k in (2, 3):
        cfg = small_cfg(E=4, H=512, I=256, k=k)
        run_and_compare(cfg, 45, overrides=dict(tile_rows=tile_rows))


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("s1,s2", [(1, 1), (2, 1), (3, 2), (5, 4)])
def test_split_k_with_nan_poisoned_workspace(s1, s2, path):
    """Split-K factors above the number of K blocks leave empty partitions;
    they must write zero partials (workspace poisoned with NaN bytes first)."""
    for act in (gen.ACT_SWIGLU, gen.ACT_RELU2):
        cfg = small_cfg(E=4, H=768, I=256, k=2, act=act)   # 3 K blocks in GEMM1, 1 in GEMM2
        split_case(cfg, s1, s2, path)


@pytest.mark.parametrize("act,inter", [(gen.ACT_SWIGLU, 512), (gen.ACT_RELU2, 1024)])
def test_tensor_core_tail_pieces(monkeypatch, act, inter):
    """More gate/up units than SMs (48 route tiles x 4 unit groups = 192 on
    152 SMs): the 40 units of the last, partial wave are cut into 2 or 3 K
    pieces (6 K blocks) whose partials the last piece to finish sums in piece
    order.  On a NaN-poisoned workspace each setting matches the oracle and
    repeats bit for bit."""
    cfg = small_cfg(E=48, H=1536, I=inter, k=4, act=act, seed=23)
    T = 96
    w, x, ids, tw = case_on_gpu(cfg, T)
    ref = oracle_rows(cfg, w, x, ids, tw)
    for pieces in ("0", "2", "4"):
        monkeypatch.setenv("W4A16_MOE_TAIL_PIECES", pieces)
        moe = make_moe(cfg, T)
        moe.set_gemm_path(PATHS["tc"])
        moe.workspace.fill_(0xFF)
        a = moe(x, w, tw, ids).clone()
        b = moe(x, w, tw, ids)
        torch.cuda.synchronize()
        moe.check_device_error()
        assert moe.read_route_layout(T)["num_tiles"] >= 40
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        compare(a, ref, f"tail pieces {pieces} act {act}")


def split_case(cfg, s1, s2, path):
    w, x, ids, tw = case_on_gpu(cfg, 9)
    moe = make_moe(cfg, 9)
    moe.set_gemm_path(PATHS[path])
    moe.set_overrides(gemm1_splits=s1, gemm2_splits=s2)
    moe.workspace.fill_(0xFF)
    out = moe(x, w, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    compare(out, oracle_rows(cfg, w, x, ids, tw), f"splits {s1},{s2} {path} act {cfg.act}")


@pytest.mark.parametrize("path", list(PATHS))
def test_all_routes_invalid_gives_exact_zero(path):
    cfg = small_cfg()
    w, x, ids, tw = case_on_gpu(cfg, 13)
    ids = torch.full_like(ids, -1)
    moe = make_moe(cfg, 13)
    moe.set_gemm_path(PATHS[path])
    moe.workspace.fill_(0xFF)
    out = moe(x, w, tw, ids)
    torch.cuda.synchronize()
    assert torch.all(out.view(torch.int16) == 0)


@pytest.mark.parametrize("path", list(PATHS))
def test_masked_ids_and_expert_offset(path):
    cfg = small_cfg(E=6, expert_offset=10)
    w, x, _, tw = case_on_gpu(cfg, 20)
    g = torch.Generator().manual_seed(5)
    ids = torch.randint(8, 18, (20, 2), generator=g, dtype=torch.int32)  # 8, 9, 16, 17: other ranks
    ids[3, 1] = -1
    moe = make_moe(cfg, 20)
    moe.set_gemm_path(PATHS[path])
    out = moe(x, w, tw, ids.cuda())
    torch.cuda.synchronize()
    compare(out, oracle_rows(cfg, w, x, ids, tw), "masked")


@pytest.mark.parametrize("path", list(PATHS))
def test_renormalize(path):
    cfg = small_cfg(k=4)
    run_and_compare(cfg, 17, renormalize=True, path=path)


@pytest.mark.parametrize("path", list(PATHS))
def test_deterministic_bitwise_and_pdl_off(monkeypatch, path):
    cfg = small_cfg(E=8, H=1024, I=256, k=4)
    w, x, ids, tw = case_on_gpu(cfg, 50)
    moe = make_moe(cfg, 50)
    moe.set_gemm_path(PATHS[path])
    outs = [moe(x, w, tw, ids).clone() for _ in range(3)]
    monkeypatch.setenv("W4A16_MOE_PDL", "0")
    moe2 = make_moe(cfg, 50)
    moe2.set_gemm_path(PATHS[path])
    outs.append(moe2(x, w, tw, ids).clone())
    moe.set_overrides(gemm1_splits=2)
    split_out = moe(x, w, tw, ids).clone()
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    compare(split_out, oracle_rows(cfg, w, x, ids, tw), "split")


@pytest.mark.parametrize("path", list(PATHS))
def test_cuda_graph_replay_with_new_inputs(path):
    cfg = small_cfg(E=8, H=1024, I=256, k=2)
    w, x, ids, tw = case_on_gpu(cfg, 33)
    moe = make_moe(cfg, 33)
    moe.set_gemm_path(PATHS[path])
    out = torch.empty(33, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        moe(x, w, tw, ids, out=out, stream=s)  # warm up on the capture stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe(x, w, tw, ids, out=out, stream=s)
    for trial in range(3):
        x2 = gen.make_activations(cfg, 33, "cuda", seed=100 + trial)
        ids2, tw2 = gen.make_routes(cfg, 33, "cuda", seed=200 + trial)
        x.copy_(x2)
        ids.copy_(ids2)
        tw.copy_(tw2)
        g.replay()
        torch.cuda.synchronize()
        eager = moe(x2, w, tw2, ids2).clone()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
        compare(out, oracle_rows(cfg, w, x2, ids2, tw2), f"graph replay {trial}")


def test_forward_host_matches_device_path():
    cfg = small_cfg()
    w, x, ids, tw = case_on_gpu(cfg, 19)
    moe = make_moe(cfg, 19)
    dev = moe(x, w, tw, ids).clone()
    torch.cuda.synchronize()
    host = moe.forward_host(x.cpu().pin_memory(), w, tw.cpu().pin_memory(), ids.cpu().pin_memory())
    assert torch.equal(host.view(torch.int16), dev.cpu().view(torch.int16))


# ---------------------------------------------------------------------------
# full-size workloads: every token count of every workload, in the launch
# configuration the benchmark times (planner's path, relaid-out weights)
# ---------------------------------------------------------------------------

FULL = [(name, T) for name, cfg in gen.CONFIGS.items() if name != gen.TINY.name for T in cfg.tokens]


def boundary_tokens(moe, ids, T, k, want=64, seed=0):
    """Tokens whose routes sit in the last route tile of their expert (one per
    expert: the token of the tile's last valid slot -- the partial tiles the
    padding logic touches), topped up with random tokens to at least `want`."""
    lay = moe.read_route_layout(T)
    perm = lay["perm"].numpy()
    tiles = lay["tiles"].numpy()
    last = {}
    for e, m0, rows, _ in tiles:
        last[int(e)] = (int(m0), int(rows))
    toks = set()
    for e, (m0, rows) in last.items():
        r = int(perm[m0 + rows - 1])
        assert r >= 0
        toks.add(r // k)
    rng = np.random.default_rng(seed)
    extra = rng.permutation(T)
    i = 0
    while len(toks) < min(want, T):
        toks.add(int(extra[i]))
        i += 1
    toks.update([0, T - 1])
    return sorted(toks)


@pytest.mark.parametrize("name,T", FULL, ids=[f"{n}-T{t}" for n, t in FULL])
def test_full_size_every_token_count(name, T):
    cfg = gen.CONFIGS[name]
    w = _full_weights(cfg)
    moe = make_moe(cfg, max(cfg.tokens))
    wi = moe.relayout_weights(w)
    _, x, ids, tw = case_on_gpu(cfg, T, weights_gpu=w)
    out = moe(x, wi, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    # repeat runs are bit-identical (also catches stale operand reads)
    again = moe(x, wi, tw, ids)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), out.view(torch.int16)), f"{name} T={T} not deterministic"
    rows = boundary_tokens(moe, ids, T, cfg.top_k, seed=T)
    assert len(rows) >= min(64, T)
    ref = oracle_rows(cfg, w, x, ids, tw, rows=rows, w_cpu=_full_weights_cpu(cfg))
    compare(out[rows], ref, f"{name} T={T} ({moe.route_info(T).gemm_path})")


@pytest.mark.parametrize("T", [8, 256, 1024])
def test_full_size_checkpoint_layout_kimi(T):
    """The checkpoint weight layout at full size, on the planner's path."""
    cfg = gen.KIMI
    w = _full_weights(cfg)
    moe = make_moe(cfg, T)
    _, x, ids, tw = case_on_gpu(cfg, T, weights_gpu=w)
    out = moe(x, w, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    rows = boundary_tokens(moe, ids, T, cfg.top_k, seed=T + 1)
    compare(out[rows], oracle_rows(cfg, w, x, ids, tw, rows=rows, w_cpu=_full_weights_cpu(cfg)), f"kimi T={T} ckpt")


_W = {}


def _full_weights(cfg):
    # one workload's weights on the device at a time (bounded device memory)
    if cfg.name not in _W:
        _W.clear()
        _W[cfg.name] = (gen.make_weights(cfg, "cuda"), None)
    return _W[cfg.name][0]


def _full_weights_cpu(cfg):
    w, wc = _W[cfg.name]
    if wc is None:
        wc = w.to("cpu")
        _W[cfg.name] = (w, wc)
    return wc
