"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: hand-built
bytes from the packing rule, library conversions, an independently written
numpy float64 MLP, exact algebraic identities, and brute force on tiny cases.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent helpers (numpy / torch library routines, not the oracle's code)
# ---------------------------------------------------------------------------

def np_nibbles_signed(b: np.ndarray, high: bool) -> np.ndarray:
    """Sign-extend a nibble by moving it to the top of an int8 and shifting
    arithmetically (hardware two's complement, a different mechanism from the
    oracle's explicit rule)."""
    b = b.astype(np.uint8)
    top = (b & np.uint8(0xF0)) if high else (b << np.uint8(4)).astype(np.uint8)
    return top.view(np.int8) >> 4


def np_dequant(cfg, packed: torch.Tensor, scales: torch.Tensor, rows: int, cols: int):
    p = packed.cpu().numpy()
    s = scales.cpu().float().numpy().astype(np.float64)
    if cfg.scale_kind == gen.SCALE_GROUP32:
        q = np.empty((rows, cols), np.float64)
        q[:, 0::2] = np_nibbles_signed(p, False)
        q[:, 1::2] = np_nibbles_signed(p, True)
        return q * np.repeat(s, 32, axis=1)
    q = np.empty((rows, cols), np.float64)
    q[0::2, :] = np_nibbles_signed(p, False)
    q[1::2, :] = np_nibbles_signed(p, True)
    return q * s[:, None]


def np_act_in(cfg, x: torch.Tensor) -> np.ndarray:
    return x.cpu().float().numpy().astype(np.float64)


def np_expert_mlp(cfg, W, x64, e):
    W1, W2 = W[e]
    h = W1 @ x64
    if cfg.act == gen.ACT_SWIGLU:
        g, u = h[: cfg.inter], h[cfg.inter:]
        a = g / (1.0 + np.exp(-g)) * u
    else:
        a = np.maximum(h, 0.0) ** 2
    return W2 @ a


def np_weights(cfg, w):
    out = []
    for e in range(cfg.num_experts):
        W1 = np_dequant(cfg, w.w13[e], w.s13[e], cfg.n1, cfg.hidden)
        W2 = np_dequant(cfg, w.w2[e], w.s2[e], cfg.hidden, cfg.inter)
        out.append((W1, W2))
    return out


def small_cfg(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16, E=3, H=64, I=64, k=2, **kw):
    return gen.MoEConfig("small", E, H, I, k, act=act, scale_kind=scale, act_dtype=dt, seed=7,
                         weight_std=0.1, **kw)


# ---------------------------------------------------------------------------
# O1: packing convention
# ---------------------------------------------------------------------------

def read_packing_golden():
    rows = []
    with open(os.path.join(GOLDEN, "int4_packing_bytes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b, h = line.split()
            rows.append((int(a), int(b), int(h, 16)))
    return rows


def test_unpack_along_k_hand_built_bytes():
    rows = read_packing_golden()
    packed = np.array([[r[2] for r in rows]], dtype=np.uint8)
    q = oracle.unpack_along_k(packed, 1, 2 * len(rows))
    want = np.array([[v for r in rows for v in (r[0], r[1])]], dtype=np.int8)
    np.testing.assert_array_equal(q, want)


def test_unpack_along_rows_hand_built_bytes():
    rows = read_packing_golden()
    packed = np.array([[r[2] for r in rows]], dtype=np.uint8)  # one row pair, many columns
    q = oracle.unpack_along_rows(packed, 2, len(rows))
    np.testing.assert_array_equal(q[0], np.array([r[0] for r in rows], np.int8))
    np.testing.assert_array_equal(q[1], np.array([r[1] for r in rows], np.int8))


def test_unpack_all_bytes_against_arithmetic_shift():
    b = np.arange(256, dtype=np.uint8)
    q = oracle.unpack_along_k(b[None, :], 1, 512)
    np.testing.assert_array_equal(q[0, 0::2], np_nibbles_signed(b, False))
    np.testing.assert_array_equal(q[0, 1::2], np_nibbles_signed(b, True))
    assert q.min() == -8 and q.max() == 7


def test_generator_packers_match_golden_bytes():
    rows = read_packing_golden()
    q = torch.tensor([[v for r in rows for v in (r[0], r[1])]], dtype=torch.int8)
    p = gen.pack_int4_along_k(q)
    assert p.tolist()[0] == [r[2] for r in rows]
    q2 = torch.tensor([[r[0] for r in rows], [r[1] for r in rows]], dtype=torch.int8)
    p2 = gen.pack_int4_along_rows(q2)
    assert p2.tolist()[0] == [r[2] for r in rows]


# ---------------------------------------------------------------------------
# Interleaved relayout of the packed weights (the layout the library's
# w4a16_moe_relayout_weights documents)
# ---------------------------------------------------------------------------

def read_relayout_golden():
    cases = []
    with open(os.path.join(GOLDEN, "interleaved_relayout.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, src, dst = (part.split() for part in line.split("|"))
            kind, n, k = (int(v) for v in head)
            cases.append((kind, n, k, bytes(int(h, 16) for h in src), bytes(int(h, 16) for h in dst)))
    return cases


def test_relayout_hand_worked_words():
    cases = read_relayout_golden()
    assert len(cases) == 4
    for kind, n, k, src, dst in cases:
        out = oracle.relayout_interleaved(np.frombuffer(src, np.uint8), kind, 1, n, k)
        assert out.tobytes() == dst, (kind, n, k, out.tobytes().hex(), dst.hex())


def test_relayout_group_and_per_channel_inputs_agree():
    """The same code matrix packed either way (the generator's two packers,
    checked against hand-built bytes above) relays out to the same bytes, and
    each 32-bit word of a row holds the multiset of that word's codes."""
    rng = np.random.default_rng(3)
    E, N, K = 3, 6, 48
    q = torch.from_numpy(rng.integers(-8, 8, size=(E, N, K)).astype(np.int8))
    along_k = torch.stack([gen.pack_int4_along_k(q[e]) for e in range(E)])
    along_rows = torch.stack([gen.pack_int4_along_rows(q[e]) for e in range(E)])
    a = oracle.relayout_interleaved(along_k, 0, E, N, K)
    b = oracle.relayout_interleaved(along_rows, 1, E, N, K)
    np.testing.assert_array_equal(a, b)
    nib = np.stack([a & 0xF, a >> 4], axis=-1).reshape(E, N, K // 8, 8)
    codes = np.sort(((nib.astype(np.int16) ^ 8) - 8), axis=-1)
    np.testing.assert_array_equal(codes, np.sort(q.numpy().reshape(E, N, K // 8, 8), axis=-1))


# ---------------------------------------------------------------------------
# O2: quantiser round trip through the oracle's dequantiser
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("group", [32, None])
def test_quantizer_round_trip(group):
    torch.manual_seed(1)
    w = torch.randn(64, 256) * 0.02
    w[3, 32:64] = 0.0       # an all-zero group
    w[5, :] = 0.0           # an all-zero row
    q, s = gen.quantize_symmetric(w, group)
    if group:
        packed = gen.pack_int4_along_k(q)
        deq = oracle.dequant(packed, s, 64, 256, gen.SCALE_GROUP32)
        s_full = s.float().repeat_interleave(32, dim=1).double().numpy()
        amax = w.view(64, 8, 32).abs().amax(2)
        qmax = q.view(64, 8, 32).abs().amax(2)
    else:
        packed = gen.pack_int4_along_rows(q)
        deq = oracle.dequant(packed, s, 64, 256, gen.SCALE_PER_CHANNEL)
        s_full = s.float()[:, None].expand(64, 256).double().numpy()
        amax = w.abs().amax(1)
        qmax = q.abs().amax(1)
    wd = w.double().numpy()
    # |w - q*s| <= s/2 for every element (the scale is absmax/7, so no element clips
    # by more than BF16 rounding of the scale allows)
    err = np.abs(wd - deq)
    assert np.all(err <= s_full * 0.5 * (1 + 2 ** -7) + 1e-30)
    # scale = absmax / 7, rounded to BF16
    s32 = s.float()
    nz = amax > 0
    rel = ((s32[nz] - amax[nz] / 7) / (amax[nz] / 7)).abs()
    assert float(rel.max()) <= 2 ** -8
    # every nonzero group/row reaches |q| = 7 at its absmax element; zero ones give 0
    assert torch.all(qmax[nz] == 7)
    assert torch.all(qmax[~nz] == 0)
    assert np.all(deq[5] == 0.0)


# ---------------------------------------------------------------------------
# 16-bit conversions against torch's library conversions
# ---------------------------------------------------------------------------

def test_fp_encoders_match_torch():
    torch.manual_seed(2)
    x = torch.cat([torch.randn(20000) * 10.0 ** torch.randint(-9, 6, (20000,)).float(),
                   torch.tensor([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, -1e9,
                                 2 ** -24, 2 ** -25, 3 * 2 ** -26, 2 ** -14, 1.0 + 2 ** -11,
                                 1.0 + 3 * 2 ** -11, float("inf"), -float("inf")])])
    xb = x.float().numpy()
    bf = oracle.bf16_encode(xb)
    tb = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bf, tb)
    fh = oracle.fp16_encode(xb)
    th = x.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(fh, th)
    dec = oracle.fp16_decode(th)
    np.testing.assert_array_equal(dec, x.to(torch.float16).double().numpy())


# ---------------------------------------------------------------------------
# O5: route preparation against numpy library routines and brute force
# ---------------------------------------------------------------------------

def np_route_layout(ids: np.ndarray, E: int, off: int, bm: int):
    flat = ids.reshape(-1).astype(np.int64)
    loc = flat - off
    valid = (flat != -1) & (loc >= 0) & (loc < E)
    counts = np.bincount(loc[valid], minlength=E)
    key = np.where(valid, loc, E)            # invalid routes sort last
    order = np.argsort(key, kind="stable")[: int(valid.sum())]
    return counts, order


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("bm", [1, 4, 16])
def test_route_prep_against_numpy(seed, bm):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 12))
    k = int(rng.choice([1, 2, 3, 4, 6, 8]))
    T = int(rng.integers(0, 40))
    off = int(rng.integers(0, 3))
    ids = rng.integers(-1, E + off + 3, size=(T, k)).astype(np.int32)
    if seed == 3:
        ids[:] = off  # everything on one expert
    if seed == 4:
        ids[:] = -1   # everything invalid
    cfg = gen.MoEConfig("r", E, 64, 64, k, expert_offset=off)
    r = oracle.prepare_routes(cfg, ids, bm)
    counts, order = np_route_layout(ids, E, off, bm)
    np.testing.assert_array_equal(r["counts"], counts)
    padded = (counts + bm - 1) // bm * bm
    np.testing.assert_array_equal(r["offs"], np.concatenate([[0], np.cumsum(padded)]))
    # unpadded stable order == numpy stable argsort by local expert
    perm = r["perm"]
    np.testing.assert_array_equal(perm[perm >= 0], order)
    # inv is the inverse of perm on valid routes, -1 elsewhere
    inv = r["inv"]
    for s, route in enumerate(perm):
        if route >= 0:
            assert inv[route] == s
    assert int((inv >= 0).sum()) == int(counts.sum())
    # tiles cover each expert's valid rows exactly
    tiles = r["tiles"]
    assert r["num_tiles"] == int(((counts + bm - 1) // bm).sum())
    for e, m0, rows, _ in tiles:
        assert r["offs"][e] <= m0 < r["offs"][e + 1]
        assert 1 <= rows <= bm
        assert np.all(perm[m0:m0 + rows] >= 0)
        assert np.all(perm[m0 + rows:m0 + bm] == -1)


def test_route_prep_brute_force_tiny():
    ids = np.array([[2, 0], [0, -1], [5, 2], [0, 0]], np.int32)  # 5 is out of range for E=3
    cfg = gen.MoEConfig("r", 3, 64, 64, 2)
    r = oracle.prepare_routes(cfg, ids, 2)
    # expert 0: routes 1, 2, 6, 7 ; expert 1: none ; expert 2: routes 0, 5
    assert r["counts"].tolist() == [4, 0, 2]
    assert r["offs"].tolist() == [0, 4, 4, 6]
    assert r["perm"].tolist() == [1, 2, 6, 7, 0, 5]
    assert r["inv"].tolist() == [4, 0, 1, -1, -1, 5, 2, 3]
    assert r["tiles"].tolist() == [[0, 0, 2, 0], [0, 2, 2, 0], [2, 4, 2, 0]]


# ---------------------------------------------------------------------------
# O3 / O7: the forward against an independently written float64 MLP
# ---------------------------------------------------------------------------

CASES = [
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_FP16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_BF16),
]


@pytest.mark.parametrize("case", CASES)
def test_top1_weight1_equals_dense_expert_mlp(case):
    cfg = small_cfg(**case, k=1)
    w = gen.make_weights(cfg)
    T = 5
    x = gen.make_activations(cfg, T)
    W = np_weights(cfg, w)
    for e in range(cfg.num_experts):
        ids = torch.full((T, 1), e, dtype=torch.int32)
        tw = torch.ones(T, 1)
        acc, _ = oracle.moe_forward(cfg, x, w, tw, ids)
        want = np.stack([np_expert_mlp(cfg, W, np_act_in(cfg, x[t]), e) for t in range(T)])
        np.testing.assert_allclose(acc, want, rtol=2e-6, atol=1e-7 * np.abs(want).max())


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("renorm", [False, True])
def test_brute_force_tiny_moe(case, renorm):
    """E=2, H=32, I=32, T=3, k=2 against straight Python loops in float64."""
    cfg = small_cfg(**case, E=2, H=32, I=32, k=2)
    w = gen.make_weights(cfg)
    x = gen.make_activations(cfg, 3)
    ids = torch.tensor([[0, 1], [1, -1], [1, 0]], dtype=torch.int32)
    tw = torch.tensor([[0.25, 0.5], [0.75, 0.125], [0.625, 0.375]], dtype=torch.float32)
    acc, out = oracle.moe_forward(cfg, x, w, tw, ids, renormalize=renorm)
    W = np_weights(cfg, w)
    xs = np_act_in(cfg, x)
    H, I, N1 = cfg.hidden, cfg.inter, cfg.n1
    for t in range(3):
        wts = tw[t].tolist()
        if renorm:
            ssum = np.float32(0)
            for j in range(2):
                ssum = np.float32(ssum + np.float32(wts[j]))
            wts = [float(np.float32(np.float32(v) / ssum)) for v in wts]
        ref = [0.0] * H
        for j in range(2):
            e = int(ids[t, j])
            if e < 0:
                continue
            W1, W2 = W[e]
            h = [sum(W1[n][c] * xs[t][c] for c in range(H)) for n in range(N1)]
            if cfg.act == gen.ACT_SWIGLU:
                a = [h[i] / (1 + math.exp(-h[i])) * h[I + i] for i in range(I)]
            else:
                a = [max(h[i], 0.0) ** 2 for i in range(I)]
            for c in range(H):
                ref[c] += wts[j] * sum(W2[c][i] * a[i] for i in range(I))
        np.testing.assert_allclose(acc[t], np.array(ref), rtol=1e-5, atol=1e-6 * max(map(abs, ref)))
    # the cast is the library's round-to-nearest-even of the FP32 accumulator
    if cfg.act_dtype == gen.DT_BF16:
        want_bits = torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        want_bits = torch.from_numpy(acc).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out, want_bits)


# ---------------------------------------------------------------------------
# O4 / O6: identities
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny_case():
    cfg = gen.TINY
    w = gen.make_weights(cfg)
    c = gen.make_case(cfg, 16, weights=w)
    return cfg, c


def test_all_routes_invalid_gives_exact_zero(tiny_case):
    cfg, c = tiny_case
    ids = torch.full_like(c["ids"], -1)
    acc, out = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], ids)
    assert np.all(acc == 0.0) and not np.any(np.signbit(acc))
    assert np.all(out == 0)


def test_masked_expert_ids_equal_invalid(tiny_case):
    cfg, c = tiny_case
    ids = c["ids"].clone()
    ids[ids == 3] = 100          # out of the local range -> masked
    ids2 = c["ids"].clone()
    ids2[ids2 == 3] = -1
    a1, _ = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], ids)
    a2, _ = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], ids2)
    np.testing.assert_array_equal(a1, a2)


def test_expert_offset_shifts_ids(tiny_case):
    cfg, c = tiny_case
    cfg2 = cfg.with_(expert_offset=40)
    ids2 = torch.where(c["ids"] >= 0, c["ids"] + 40, c["ids"])
    a1, _ = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], c["ids"])
    a2, _ = oracle.moe_forward(cfg2, c["x"], c["weights"], c["topk_weights"], ids2)
    np.testing.assert_array_equal(a1, a2)


def test_routing_weight_scaling_is_linear(tiny_case):
    cfg, c = tiny_case
    a1, _ = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], c["ids"])
    a2, _ = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"] * 4.0, c["ids"])
    np.testing.assert_array_equal(a2, a1 * 4.0)  # power-of-two scaling is exact in FP32


def test_token_permutation_permutes_rows(tiny_case):
    cfg, c = tiny_case
    p = torch.randperm(16, generator=torch.Generator().manual_seed(3))
    a1, _ = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], c["ids"])
    a2, _ = oracle.moe_forward(cfg, c["x"][p], c["weights"], c["topk_weights"][p], c["ids"][p])
    np.testing.assert_array_equal(a2, a1[p.numpy()])


def test_row_subset_matches_full(tiny_case):
    cfg, c = tiny_case
    a1, o1 = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], c["ids"])
    rows = [15, 0, 7]
    a2, o2 = oracle.moe_forward(cfg, c["x"], c["weights"], c["topk_weights"], c["ids"], rows=rows)
    np.testing.assert_array_equal(a2, a1[rows])
    np.testing.assert_array_equal(o2, o1[rows])


def test_duplicate_route_equals_summed_weight(tiny_case):
    cfg, c = tiny_case
    ids = torch.tensor([[1, 1]] * 4, dtype=torch.int32)
    tw = torch.tensor([[0.25, 0.5]] * 4)
    ids1 = torch.tensor([[1, -1]] * 4, dtype=torch.int32)
    tw1 = torch.tensor([[0.75, 0.0]] * 4)
    x = c["x"][:4]
    a, _ = oracle.moe_forward(cfg, x, c["weights"], tw, ids)
    b, _ = oracle.moe_forward(cfg, x, c["weights"], tw1, ids1)
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7 * np.abs(b).max())


def test_renormalize_zero_sum_gives_zero(tiny_case):
    cfg, c = tiny_case
    tw = torch.zeros_like(c["topk_weights"])
    a, o = oracle.moe_forward(cfg, c["x"], c["weights"], tw, c["ids"], renormalize=True)
    assert np.all(a == 0.0)


def test_tiny_workload_has_the_two_forced_invalid_routes(tiny_case):
    cfg, c = tiny_case
    assert int(c["ids"][0, 1]) == -1 and int(c["ids"][5, 0]) == -1
    assert int((c["ids"] == -1).sum()) == 2


# ---------------------------------------------------------------------------
# masked-count layout (expert-major rows + counts): routes and forward
# ---------------------------------------------------------------------------

def test_masked_routes_structure():
    """Per expert: a prefix of clamp(counts[e], 0, max_rows) valid rows routed to
    the expert's global id, the rest invalid; every weight 1."""
    counts = np.array([0, 3, 7, 5, -2, 9], np.int32)
    M, off = 5, 40
    ids, w = oracle.masked_routes(counts, M, off)
    assert ids.shape == (len(counts) * M, 1)
    assert (w == 1.0).all()
    for e, c in enumerate(counts):
        rows = ids[e * M:(e + 1) * M, 0]
        n = min(max(int(c), 0), M)
        assert (rows[:n] == off + e).all() and (rows[n:] == -1).all()


@pytest.mark.parametrize("case", CASES[:3])
def test_masked_forward_equals_dense_expert_mlp(case):
    """Every valid row equals its expert's MLP from an independently written
    float64 evaluation; rows past an expert's count are exact zeros."""
    cfg = small_cfg(**case, E=3, k=1)
    w = gen.make_weights(cfg)
    M = 4
    counts = np.array([2, 0, 4], np.int32)
    x = gen.make_activations(cfg, cfg.num_experts * M)
    acc, _ = oracle.masked_forward(cfg, x, w, counts, M)
    W = np_weights(cfg, w)
    for e in range(cfg.num_experts):
        for i in range(M):
            r = e * M + i
            if i < counts[e]:
                want = np_expert_mlp(cfg, W, np_act_in(cfg, x[r]), e)
                np.testing.assert_allclose(acc[r], want, rtol=2e-6, atol=1e-7 * np.abs(want).max())
            else:
                assert (acc[r] == 0.0).all()
