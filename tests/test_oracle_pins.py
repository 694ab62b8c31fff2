"""Pins of the CPU oracle against things other than itself: worked examples,
library routines, closed forms, invariants and brute force (no GPU)."""
import math
import os

import numpy as np
import pytest
import torch

import workloads as WL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield [c.strip() for c in ln.split("|")]


# ---------------------------------------------------------------- e4m3 ----

def test_e4m3_decode_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([orc.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert np.array_equal(ref[~nan], mine[~nan])


def test_e4m3_golden_examples(orc):
    for val, code in _lines("e4m3_examples.txt"):
        got = int(orc.e4m3_encode([float(val)])[0])
        assert got == int(code, 16), (val, hex(got), code)


def test_e4m3_encode_matches_torch_cast_in_range(orc):
    rng = np.random.default_rng(0)
    # every code value, every midpoint between neighbours, and random values
    vals = np.array([orc.e4m3_value(c) for c in range(0x7f)])
    mids = (vals[:-1] + vals[1:]) / 2
    rand = np.concatenate([rng.normal(0, s, 4000) for s in (1e-3, 0.1, 1, 30, 150)])
    x = np.concatenate([vals, mids, -vals, -mids, rand]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(x)
    # +0 / -0 both encode zero; torch keeps the sign like the oracle does
    assert np.array_equal(ref, got), np.flatnonzero(ref != got)[:10]


def test_e4m3_saturates(orc):
    got = orc.e4m3_encode([449.0, 463.9, 464.0, 1e6, -1e30])
    assert list(got) == [0x7e, 0x7e, 0x7e, 0x7e, 0xfe]


# -------------------------------------------------------------- router ----

def test_route_golden_examples(orc):
    for kind, E, topk, ng, tg, rn, logits, bias, ids, w in _lines("route_examples.txt"):
        E, topk, ng, tg, rn = int(E), int(topk), int(ng), int(tg), int(rn)
        lg = np.array([float(v) for v in logits.split()], np.float32).reshape(1, E)
        b = None if bias == "-" else np.array([float(v) for v in bias.split()], np.float32)
        fn = orc.SOFTMAX if kind == "softmax" else orc.SIGMOID
        gi, gw, _ = orc.route(lg, b, topk, fn, ng, tg, bool(rn))
        assert list(gi[0]) == [int(v) for v in ids.split()], (kind, logits, gi)
        np.testing.assert_allclose(gw[0], [float(v) for v in w.split()], atol=2e-7)


def test_route_softmax_topk_is_stable_argsort(orc):
    rng = np.random.default_rng(1)
    for E, topk in ((8, 2), (64, 6), (256, 8)):
        lg = rng.standard_normal((300, E)).astype(np.float32)
        lg[:20, :] = np.round(lg[:20, :])  # many exact ties
        ids, w, _ = orc.route(lg, None, topk, orc.SOFTMAX)
        ref = np.argsort(-lg, axis=1, kind="stable")[:, :topk]
        assert np.array_equal(ids, ref)
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)
        if topk == 2:  # closed form of a renormalised top-2 softmax
            l0 = np.take_along_axis(lg, ids[:, :1], 1)[:, 0].astype(np.float64)
            l1 = np.take_along_axis(lg, ids[:, 1:2], 1)[:, 0].astype(np.float64)
            np.testing.assert_allclose(w[:, 0], 1 / (1 + np.exp(l1 - l0)), rtol=1e-12)
        # unrenormalised weights are the softmax probabilities themselves
        _, wp, _ = orc.route(lg, None, topk, orc.SOFTMAX, renorm=False)
        p = torch.softmax(torch.from_numpy(lg).double(), 1).numpy()
        np.testing.assert_allclose(wp, np.take_along_axis(p, ids, 1), rtol=1e-12)


def test_route_sigmoid_one_group_is_argsort_of_logit_plus_bias(orc):
    rng = np.random.default_rng(2)
    E, topk = 256, 8
    lg = rng.standard_normal((200, E)).astype(np.float32)
    b = rng.uniform(-3, 0, E).astype(np.float32)
    ids, w, _ = orc.route(lg, b, topk, orc.SIGMOID, 1, 1)
    v = (lg + b).astype(np.float32)
    # the sigmoid is increasing: the top-k by score is the top-k by l + b
    ref = np.argsort(-v, axis=1, kind="stable")[:, :topk]
    assert np.array_equal(ids, ref)
    s = 1 / (1 + np.exp(-v.astype(np.float64)))
    sel = np.take_along_axis(s, ids, 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12)


def test_route_sigmoid_grouped_invariants(orc):
    """Every choice of the group-limited router is valid: kept groups have
    keys no smaller than dropped ones, all ids lie in kept groups, and no
    eligible unchosen expert scores above a chosen one."""
    cfg = WL.SMALL_SIGMOID
    d = WL.make_inputs(cfg)
    lg, b = d["logits"].numpy(), d["bias"].numpy()
    ids, w, margin = orc.route(lg, b, cfg.topk, orc.SIGMOID, cfg.n_groups, cfg.topk_groups)
    E, G, tg, k = cfg.E, cfg.n_groups, cfg.topk_groups, cfg.topk
    gs = E // G
    s = (1 / (1 + np.exp(-(lg + b).astype(np.float32).astype(np.float64))))
    for t in range(cfg.M):
        key = np.sort(s[t].reshape(G, gs), 1)[:, -2:].sum(1)
        kept = set(np.argsort(-key, kind="stable")[:tg].tolist())
        chosen_groups = set(int(e) // gs for e in ids[t])
        assert len(set(ids[t].tolist())) == k
        # every chosen expert sits in one of the best topk_groups groups
        # (a group tied with the weakest kept one may stand in for it)
        kth = np.sort(key)[::-1][tg - 1]
        assert all(key[g] >= kth - 1e-6 for g in chosen_groups)
        chosen_min = s[t, ids[t]].min()
        for e in range(E):
            if e // gs in kept and e not in ids[t]:
                assert s[t, e] <= chosen_min + 1e-6
        assert np.all(np.diff(s[t, ids[t]]) <= 1e-7)  # descending order
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-12)
    assert np.all(margin >= -1e-6)


# ------------------------------------------------------ count / permute ----

def test_count_matches_bincount_and_sums_to_P(orc):
    rng = np.random.default_rng(3)
    for E, P in ((8, 128), (256, 65536), (32, 7)):
        ids = rng.integers(0, E, P).astype(np.int32)
        c, bad = orc.count(ids, E)
        assert bad == 0
        assert np.array_equal(c, np.bincount(ids, minlength=E))
        assert c.sum() == P
    ids = np.array([0, 5, -1, 3, 9, 3], np.int32)
    c, bad = orc.count(ids, 4)
    assert bad == 3 and list(c) == [1, 0, 0, 2]


def test_align_is_stable_argsort_and_inverse(orc):
    rng = np.random.default_rng(4)
    for E, M, k in ((8, 64, 2), (256, 1000, 8), (4, 3, 1)):
        ids = rng.integers(0, E, (M, k)).astype(np.int32)
        off, srt, inv = orc.align(ids, E)
        flat = ids.ravel()
        assert np.array_equal(srt, np.argsort(flat, kind="stable"))
        assert off[0] == 0 and off[E] == M * k
        assert np.array_equal(np.diff(off), np.bincount(flat, minlength=E))
        assert np.array_equal(inv[srt], np.arange(M * k))
        assert np.array_equal(srt[inv], np.arange(M * k))
        for e in range(E):
            assert np.all(flat[srt[off[e]:off[e + 1]]] == e)


def test_permute_then_unpermute_is_identity(orc):
    """Identity experts with weights summing to 1 give back the input."""
    rng = np.random.default_rng(5)
    M, K, E, k = 50, 24, 8, 3
    x = rng.standard_normal((M, K))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    w = rng.uniform(0.1, 1, (M, k))
    w /= w.sum(1, keepdims=True)
    off, srt, inv = orc.align(ids, E)
    xp = orc.permute_rows(x, srt, k)
    out = orc.unpermute_reduce(xp, inv, w)
    np.testing.assert_allclose(out, x, rtol=1e-12, atol=1e-12)
    # a non-identity expert: scaling every permuted row by 2 doubles the output
    out2 = orc.unpermute_reduce(2 * xp, inv, w)
    np.testing.assert_allclose(out2, 2 * x, rtol=1e-12, atol=1e-12)


# -------------------------------------------------------------- quant ----

def _bits(t):
    return WL.bf16_bits(t)


def test_quant_group_codes_are_torch_cast_and_max_maps_to_448(orc):
    g = torch.Generator().manual_seed(6)
    x = (torch.randn(37, 512, generator=g) * torch.logspace(-3, 2, 512)).to(torch.bfloat16)
    x[3, :128] = 0  # an all-zero group
    q, s = orc.quant_fp8_group(_bits(x), 128)
    xf = x.float().view(37, 4, 128)
    amax = xf.abs().amax(-1)
    # the group's largest magnitude lands on the top code
    top = torch.from_numpy(q).view(37, 4, 128)[torch.arange(37)[:, None], torch.arange(4)[None], xf.abs().argmax(-1)]
    nz = amax > 0
    assert torch.all((top[nz] & 0x7f) == 0x7e)
    # codes are the library cast of x / s
    sf = torch.from_numpy(s).view(37, 4, 1)
    ref = (xf / sf).to(torch.float8_e4m3fn).view(torch.uint8).view(37, 512).numpy()
    assert np.array_equal(q, ref)
    # dequantisation error bound of a 3-bit mantissa (2^-4 relative; 2^-10 s
    # absolute in the subnormal range)
    deq = torch.from_numpy(q).view(torch.float8_e4m3fn).double().view(37, 4, 128) * sf.double()
    err = (deq - xf.double()).abs()
    bound = torch.maximum(xf.double().abs() * 2.0 ** -4, sf.double() * 2.0 ** -10)
    assert torch.all(err <= bound * (1 + 1e-9))
    assert q[3, :128].max() == 0 and s[3, 0] == np.float32(1e-12) / np.float32(448)


def test_quant_block_is_per_tile_group_quant(orc):
    g = torch.Generator().manual_seed(7)
    w = (torch.randn(256, 384, generator=g) * 0.05).to(torch.bfloat16)
    q, s = orc.quant_fp8_block(_bits(w), 128)
    assert s.shape == (2, 3)
    wf = w.float()
    for br in range(2):
        for bc in range(3):
            tile = wf[br * 128:(br + 1) * 128, bc * 128:(bc + 1) * 128]
            assert s[br, bc] == np.float32(tile.abs().max().item()) / np.float32(448)
            ref = (tile / float(s[br, bc])).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(q[br * 128:(br + 1) * 128, bc * 128:(bc + 1) * 128], ref)


# ------------------------------------------------------------- experts ----

def _silu(z):
    return z / (1 + np.exp(-z))


def test_single_expert_is_dense_swiglu_mlp(orc):
    """E = 1, topk = 1: the layer is a dense SwiGLU MLP, checked against
    fp64 numpy matmuls (rows [0, N) of w1 are the gate, [N, 2N) the up)."""
    cfg = WL.MoEConfig("e1", M=9, K=64, N=32, E=1, topk=1, seed=21)
    d = WL.make_inputs(cfg)
    W = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"]))
    out, ids, w = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1,
                                  orc.SOFTMAX, W)
    x = d["x"].double().numpy()
    w1 = d["w1"][0].double().numpy()
    w2 = d["w2"][0].double().numpy()
    h = _silu(x @ w1[:32].T) * (x @ w1[32:].T)
    ref = h @ w2.T
    assert np.all(ids == 0) and np.all(w == 1.0)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    hh, yy = orc.expert_row(_bits(d["x"]), 4, 0, W)
    np.testing.assert_allclose(hh, h[4], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(yy, ref[4], rtol=1e-10, atol=1e-13)


def test_layer_equals_per_expert_batched_loop(orc):
    """Two routes to one answer: the oracle's per-token loop against a
    per-expert loop of numpy matmuls over gathered tokens."""
    cfg = WL.SMALL_BF16
    cfg = WL.MoEConfig("pe", M=40, K=128, N=64, E=8, topk=3, seed=22)
    d = WL.make_inputs(cfg)
    W = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"]))
    out, ids, w = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None,
                                  cfg.topk, orc.SOFTMAX, W)
    x = d["x"].double().numpy()
    ref = np.zeros_like(out)
    for e in range(cfg.E):
        t, j = np.nonzero(ids == e)
        if t.size == 0:
            continue
        w1 = d["w1"][e].double().numpy()
        w2 = d["w2"][e].double().numpy()
        y = (_silu(x[t] @ w1[:cfg.N].T) * (x[t] @ w1[cfg.N:].T)) @ w2.T
        np.add.at(ref, t, w[t, j][:, None] * y)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    # linearity in w2: doubling w2 doubles the output exactly
    W2 = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"] * 2))
    out2, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None,
                                 cfg.topk, orc.SOFTMAX, W2)
    np.testing.assert_array_equal(out2, 2 * out)
    # a listed subset of tokens gives exactly the rows of the full run
    sub, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None,
                                cfg.topk, orc.SOFTMAX, W, tokens=[7, 0, 39])
    np.testing.assert_array_equal(sub, out[[7, 0, 39]])


def test_fp8_single_expert_is_dequantised_swiglu(orc):
    """FP8: with E = 1 the layer is the dense SwiGLU MLP of the dequantised
    operands (library cast of the codes times the block scales)."""
    cfg = WL.MoEConfig("f8", M=6, K=256, N=128, E=1, topk=1, dtype=WL.FP8, seed=23)
    d = WL.make_inputs(cfg)
    q1, s1 = orc.quant_fp8_block(_bits(d["w1"][0]))
    q2, s2 = orc.quant_fp8_block(_bits(d["w2"][0]))
    W = orc.Weights(orc.FP8, q1[None], q2[None], s1[None], s2[None])
    out, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1,
                                orc.SOFTMAX, W, requant_h=False)

    def deq(q, s, rows, cols):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
        return v * np.kron(s.astype(np.float64), np.ones((rows, cols)))

    qx, sx = orc.quant_fp8_group(_bits(d["x"]))
    x = deq(qx, sx, 1, 128)
    w1 = deq(q1, s1, 128, 128)
    w2 = deq(q2, s2, 128, 128)
    h = _silu(x @ w1[:128].T) * (x @ w1[128:].T)
    np.testing.assert_allclose(out, h @ w2.T, rtol=1e-10, atol=1e-12)
    # with requantisation of h, each 128-group of h goes through the same
    # quantiser; check h of one row against the library cast
    hq, _ = orc.expert_row(_bits(d["x"]), 2, 0, W, requant_h=True)
    h32 = h[2].astype(np.float32)
    s = np.float32(np.abs(h32).max()) / np.float32(448)
    ref = torch.from_numpy(h32 / s).to(torch.float8_e4m3fn).double().numpy() * float(s)
    np.testing.assert_allclose(hq, ref, rtol=0, atol=float(s) * 2 ** -3 + 1e-12)
    assert np.mean(np.abs(hq - ref) < 1e-12) > 0.99


def test_batched_equals_standard_on_the_same_routing(orc):
    """BatchedExperts rows computed by the oracle equal the Standard layer's
    unweighted expert outputs when x_b is built from the Standard permutation;
    padded rows are never written."""
    cfg = WL.MoEConfig("bs", M=30, K=128, N=128, E=4, topk=1, seed=24)
    d = WL.make_inputs(cfg)
    W = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"]))
    out, ids, w = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1,
                                  orc.SOFTMAX, W)
    assert np.all(w == 1.0)
    off, srt, inv = orc.align(ids, cfg.E)
    T = 16
    counts = np.minimum(np.diff(off), T).astype(np.int32)
    xb = torch.full((cfg.E, T, cfg.K), 77.0, dtype=torch.bfloat16)
    for e in range(cfg.E):
        for r in range(counts[e]):
            xb[e, r] = d["x"][srt[off[e] + r]]
    yb, n = orc.batched_experts(_bits(xb), counts, W)
    assert n == counts.sum()
    for e in range(cfg.E):
        for r in range(T):
            if r < counts[e]:
                np.testing.assert_allclose(yb[e, r], out[srt[off[e] + r]], rtol=1e-12, atol=1e-14)
            else:
                assert np.all(np.isnan(yb[e, r]))


def test_fp8_batched_rows_are_dequantised_swiglu_with_requantised_h(orc):
    """FP8 BatchedExperts: each valid row (e, r) is expert e's SwiGLU of the
    dequantised row (1 x 128 group scales) and dequantised weights (128 x 128
    block scales), with h requantised per 128-group by the library e4m3 cast
    before the down projection; padded rows are never written."""
    E, T, K, N = 3, 5, 256, 256
    rng = np.random.default_rng(31)
    xb = torch.from_numpy(rng.standard_normal((E, T, K)).astype(np.float32)).to(torch.bfloat16)
    w1 = torch.from_numpy((rng.standard_normal((E, 2 * N, K)) / np.sqrt(K)).astype(np.float32)).to(torch.bfloat16)
    w2 = torch.from_numpy((rng.standard_normal((E, K, N)) / np.sqrt(N)).astype(np.float32)).to(torch.bfloat16)
    q1, s1, q2, s2 = [], [], [], []
    for e in range(E):
        a, b = orc.quant_fp8_block(_bits(w1[e])); q1.append(a); s1.append(b)
        a, b = orc.quant_fp8_block(_bits(w2[e])); q2.append(a); s2.append(b)
    W = orc.Weights(orc.FP8, np.stack(q1), np.stack(q2), np.stack(s1), np.stack(s2))
    counts = np.array([5, 0, 2], np.int32)
    yb, n = orc.batched_experts(_bits(xb), counts, W, requant_h=True)
    assert n == 7

    def deq(q, s, rows, cols):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
        return v * np.kron(s.astype(np.float64), np.ones((rows, cols)))

    for e in range(E):
        wd1 = deq(q1[e], s1[e], 128, 128)
        wd2 = deq(q2[e], s2[e], 128, 128)
        for r in range(T):
            if r >= counts[e]:
                assert np.all(np.isnan(yb[e, r]))
                continue
            qx, sx = orc.quant_fp8_group(_bits(xb[e, r:r + 1]))
            x = deq(qx, sx, 1, 128)[0]
            h = (_silu(x @ wd1[:N].T) * (x @ wd1[N:].T)).astype(np.float32)
            hq = np.empty(N)
            for g in range(N // 128):
                hg = h[g * 128:(g + 1) * 128]
                sc = np.float32(np.abs(hg).max()) / np.float32(448)
                hq[g * 128:(g + 1) * 128] = (torch.from_numpy(hg / sc).to(torch.float8_e4m3fn)
                                             .double().numpy() * float(sc))
            ref = hq @ wd2.T
            np.testing.assert_allclose(yb[e, r], ref, rtol=0, atol=1e-10 * np.abs(ref).max())


# ------------------------------------------- expert_map / weight on input ----

def _swiglu_np(x, w1, w2, N):
    return (_silu(x @ w1[:N].T) * (x @ w1[N:].T)) @ w2.T


def test_count_align_with_expert_map_match_numpy(orc):
    rng = np.random.default_rng(30)
    Eg, El, P = 16, 5, 3000
    emap = np.full(Eg, -1, np.int32)
    local_globals = np.array([2, 3, 7, 11, 15])
    emap[local_globals] = np.arange(El)
    ids = rng.integers(0, Eg, P).astype(np.int32)
    ids[:3] = [-1, 16, 99]  # invalid ids
    c, bad = orc.count(ids, Eg, emap, El)
    off, srt, inv = orc.align(ids, Eg, emap, El)
    ok = (ids >= 0) & (ids < Eg)
    lid = np.where(ok, emap[np.clip(ids, 0, Eg - 1)], -1)
    assert bad == 3
    assert np.array_equal(c, np.bincount(lid[lid >= 0], minlength=El))
    keep = np.flatnonzero(lid >= 0)
    assert np.array_equal(srt, keep[np.argsort(lid[keep], kind="stable")])
    assert np.all(inv[lid < 0] == -1)
    assert np.array_equal(srt[inv[keep]], keep)
    # the identity map is the same as no map
    ident = np.arange(Eg, dtype=np.int32)
    assert np.array_equal(orc.align(ids, Eg, ident, Eg)[1], orc.align(ids, Eg)[1])


def test_forward_with_expert_map_is_the_local_part_of_the_layer(orc):
    """A shard holding experts {1, 4, 6} of 8: its output is the weighted sum
    over the routed slots whose expert is local (numpy per-expert loop)."""
    cfg = WL.MoEConfig("ep", M=37, K=128, N=64, E=8, topk=3, seed=31)
    d = WL.make_inputs(cfg)
    local = [1, 4, 6]
    emap = np.full(8, -1, np.int32)
    emap[local] = np.arange(3)
    Wl = orc.Weights(orc.BF16, _bits(d["w1"][local]), _bits(d["w2"][local]))
    out, ids, w = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 3,
                                  orc.SOFTMAX, Wl, expert_map=emap)
    x = d["x"].double().numpy()
    ref = np.zeros_like(out)
    for g in local:
        t, j = np.nonzero(ids == g)
        y = _swiglu_np(x[t], d["w1"][g].double().numpy(), d["w2"][g].double().numpy(), cfg.N)
        np.add.at(ref, t, w[t, j][:, None] * y)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    # every expert local through the identity map: the plain layer
    Wg = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"]))
    full, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 3, orc.SOFTMAX, Wg)
    same, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 3, orc.SOFTMAX, Wg,
                                 expert_map=np.arange(8, dtype=np.int32))
    np.testing.assert_array_equal(full, same)


def test_weight_on_input_scales_the_expert_input(orc):
    """apply_router_weight_on_input, top-1, unrenormalised softmax weight p:
    out[t] = expert(p * x[t]) (numpy), which differs from p * expert(x[t])."""
    cfg = WL.MoEConfig("woi", M=29, K=128, N=64, E=4, topk=1, renorm=False, seed=32)
    d = WL.make_inputs(cfg)
    W = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"]))
    out, ids, w = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1,
                                  orc.SOFTMAX, W, renorm=False, weight_on_input=True)
    assert np.all(w < 1.0)
    x = d["x"].double().numpy()
    ref = np.zeros_like(out)
    for e in range(4):
        t = np.flatnonzero(ids[:, 0] == e)
        xin = x[t] * w[t, 0].astype(np.float32).astype(np.float64)[:, None]
        ref[t] = _swiglu_np(xin, d["w1"][e].double().numpy(), d["w2"][e].double().numpy(), cfg.N)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    plain, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1,
                                  orc.SOFTMAX, W, renorm=False)
    assert np.abs(plain - out).max() > 1e-3 * np.abs(out).max()


def test_quant_with_row_weights_is_cast_of_the_fp32_product(orc):
    g = torch.Generator().manual_seed(33)
    x = torch.randn(17, 256, generator=g).to(torch.bfloat16)
    rw = torch.rand(17, generator=g).to(torch.float32)
    q, s = orc.quant_fp8_group(_bits(x), row_weights=rw.numpy())
    v = (x.float() * rw[:, None]).view(17, 2, 128)
    assert np.array_equal(s, (v.abs().amax(-1) / 448.0).numpy())
    ref = (v / torch.from_numpy(s).view(17, 2, 1)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(q, ref.view(17, 256).numpy())


def test_gelu_experts_are_dense_geglu(orc):
    """activation "gelu" (gelu_and_mul): h = gelu(gate) * up with the exact
    erf GELU, checked against torch's gelu on a dense E = 1 layer."""
    cfg = WL.MoEConfig("gelu", M=11, K=64, N=32, E=1, topk=1, seed=34)
    d = WL.make_inputs(cfg)
    W = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"]), act=orc.GELU)
    out, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1, orc.SOFTMAX, W)
    x = d["x"].double()
    w1 = d["w1"][0].double()
    h = torch.nn.functional.gelu(x @ w1[:32].T) * (x @ w1[32:].T)
    ref = (h @ d["w2"][0].double().T).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    Ws = orc.Weights(orc.BF16, _bits(d["w1"]), _bits(d["w2"]))
    silu, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1, orc.SOFTMAX, Ws)
    assert np.abs(silu - out).max() > 1e-3 * np.abs(out).max()


def _rowwise_quant_torch(a32):
    """Per-row e4m3 quantisation written with numpy and torch's cast:
    s = max(amax, 1e-12) / 448 in fp32, codes = cast of the fp32 quotient."""
    a32 = np.asarray(a32, np.float32)
    s = (np.maximum(np.abs(a32).max(axis=1), np.float32(1e-12)) / np.float32(448)).astype(np.float32)
    q = torch.from_numpy(a32 / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q, s


def test_fp8_channel_quant_is_one_group_per_row(orc):
    """Per-token activations and per-channel weights: the group rule with a
    group as wide as the row equals the per-row formula and torch's cast."""
    g = torch.Generator().manual_seed(41)
    x = (torch.randn((7, 384), generator=g) * torch.linspace(0.01, 30, 384)).to(torch.bfloat16)
    q, s = orc.quant_fp8_group(_bits(x), group=384)
    qr, sr = _rowwise_quant_torch(x.float().numpy())
    assert s.shape == (7, 1)
    np.testing.assert_array_equal(s[:, 0], sr)
    np.testing.assert_array_equal(q, qr)


def test_fp8_channel_single_expert_is_dequantised_swiglu(orc):
    """FP8 with one scale per token and per weight row: with E = 1 the layer
    is the dense SwiGLU MLP of the dequantised operands; with requantisation
    the hidden row goes to bf16 and then through one scale over its N
    values (the per-row rule applied by torch's casts)."""
    cfg = WL.MoEConfig("f8c", M=6, K=256, N=256, E=1, topk=1, seed=25)  # N > 128: a row is not one 128-group
    d = WL.make_inputs(cfg)
    q1, s1 = _rowwise_quant_torch(d["w1"][0].float().numpy())
    q2, s2 = _rowwise_quant_torch(d["w2"][0].float().numpy())
    W = orc.Weights(orc.FP8_CHANNEL, q1[None], q2[None], s1[None], s2[None])

    def deq(q, s):
        return torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy() * s.astype(np.float64)[:, None]

    qx, sx = _rowwise_quant_torch(d["x"].float().numpy())
    x = deq(qx, sx)
    w1, w2 = deq(q1, s1), deq(q2, s2)
    N = cfg.N
    h = _silu(x @ w1[:N].T) * (x @ w1[N:].T)
    out, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1,
                                orc.SOFTMAX, W, requant_h=False)
    np.testing.assert_allclose(out, h @ w2.T, rtol=1e-10, atol=1e-12)

    hb = torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16).float().numpy()
    qh, sh = _rowwise_quant_torch(hb)
    hd = deq(qh, sh)
    for t in (0, 3, 5):
        hq, y = orc.expert_row(_bits(d["x"]), t, 0, W, requant_h=True)
        assert np.mean(np.abs(hq - hd[t]) <= 1e-12) > 0.99
        np.testing.assert_allclose(hq, hd[t], rtol=0, atol=float(sh[t]) * 2 ** -3 + 1e-12)
        ref = hd[t] @ w2.T
        np.testing.assert_allclose(y, ref, rtol=0, atol=2e-3 * np.abs(ref).max())


def test_fp8_tensor_quant_is_one_group_for_the_whole_tensor(orc):
    """Per-tensor activation scale: the max over every element (of the fp32
    product with the row weights), codes = torch's cast of the quotient."""
    g = torch.Generator().manual_seed(44)
    x = (torch.randn((9, 256), generator=g) * torch.linspace(0.1, 5, 9)[:, None]).to(torch.bfloat16)
    rw = (torch.rand(9, generator=g) + 0.1).numpy().astype(np.float32)
    for w in (None, rw):
        v = x.float().numpy() * (1.0 if w is None else w[:, None])
        v = v.astype(np.float32)
        s = np.float32(max(np.abs(v).max(), np.float32(1e-12))) / np.float32(448)
        q, sc = orc.quant_fp8_tensor(_bits(x), row_weights=w)
        assert sc == s
        np.testing.assert_array_equal(
            q, torch.from_numpy(v / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_fp8_tensor_layer_uses_one_scale_for_all_hidden_rows(orc):
    """Per-tensor activations (two experts, top-1): x quantised with one scale,
    every routed hidden row rounded to bf16, then one scale for all of H;
    written with numpy, torch's casts and the routing's argmax."""
    cfg = WL.MoEConfig("f8t", M=10, K=256, N=256, E=2, topk=1, seed=26)
    d = WL.make_inputs(cfg)
    N = cfg.N
    q1, s1, q2, s2 = [], [], [], []
    for e in range(2):
        a, b = _rowwise_quant_torch(d["w1"][e].float().numpy())
        c, dd = _rowwise_quant_torch(d["w2"][e].float().numpy())
        q1.append(a); s1.append(b); q2.append(c); s2.append(dd)
    W = orc.Weights(orc.FP8_TENSOR, np.stack(q1), np.stack(q2), np.stack(s1), np.stack(s2))
    out, ids, w = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1, orc.SOFTMAX,
                                  W, requant_h=True)
    ref_ids = np.argmax(d["logits"].numpy(), axis=1)
    assert np.array_equal(ids[:, 0], ref_ids)

    def deq(q, s):
        return torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy() * s

    x32 = d["x"].float().numpy()
    sx = np.float32(np.abs(x32).max()) / np.float32(448)
    xd = deq(torch.from_numpy(x32 / sx).to(torch.float8_e4m3fn).view(torch.uint8).numpy(), float(sx))
    hs = []
    for t in range(cfg.M):
        e = ref_ids[t]
        w1d = deq(q1[e], s1[e].astype(np.float64)[:, None])
        g_, u_ = xd[t] @ w1d[:N].T, xd[t] @ w1d[N:].T
        hs.append(_silu(g_) * u_)
    hb = torch.from_numpy(np.stack(hs).astype(np.float32)).to(torch.bfloat16).float().numpy()
    sh = np.float32(np.abs(hb).max()) / np.float32(448)
    hd = deq(torch.from_numpy(hb / sh).to(torch.float8_e4m3fn).view(torch.uint8).numpy(), float(sh))
    ref = np.stack([hd[t] @ deq(q2[ref_ids[t]], s2[ref_ids[t]].astype(np.float64)[:, None]).T
                    for t in range(cfg.M)])
    np.testing.assert_allclose(out, ref, rtol=0, atol=2e-3 * np.abs(ref).max())


def _clamped_cast(v32, s):
    """e4m3 codes of v / s saturating at +-448: numpy's fp32 quotient,
    clamped, then torch's cast (which itself saturates only up to 464)."""
    qv = np.clip((v32 / np.float32(s)).astype(np.float32), -448.0, 448.0)
    return torch.from_numpy(qv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_fp8_tensor_static_quant_is_the_clamped_cast(orc):
    """Static per-tensor activation scale (the quant config's a1_scale): the
    codes of x / s for the given s, values beyond 448 s saturating; with s
    the tensor's own max / 448 they are the dynamic quantiser's codes."""
    g = torch.Generator().manual_seed(45)
    x = (torch.randn((9, 256), generator=g) * torch.linspace(0.1, 5, 9)[:, None]).to(torch.bfloat16)
    rw = (torch.rand(9, generator=g) + 0.1).numpy().astype(np.float32)
    for w in (None, rw):
        v = (x.float().numpy() * (1.0 if w is None else w[:, None])).astype(np.float32)
        s_dyn = np.float32(np.abs(v).max()) / np.float32(448)
        for s in (s_dyn, s_dyn * np.float32(0.25), s_dyn * np.float32(3.0)):
            q, sc = orc.quant_fp8_tensor(_bits(x), row_weights=w, scale=s)
            assert sc == np.float32(s)
            np.testing.assert_array_equal(q, _clamped_cast(v, s))
        # a quarter of the dynamic scale saturates the largest values
        q, _ = orc.quant_fp8_tensor(_bits(x), row_weights=w, scale=s_dyn * np.float32(0.25))
        assert np.any((q & 0x7f) == 0x7e)
        qd, sd = orc.quant_fp8_tensor(_bits(x), row_weights=w)
        qs, _ = orc.quant_fp8_tensor(_bits(x), row_weights=w, scale=sd)
        np.testing.assert_array_equal(qs, qd)


def test_fp8_tensor_static_layer_uses_the_given_scales(orc):
    """Static per-tensor activation scales a1 (for x) and a2 (for H), two
    experts, top-1: x coded with a1, every routed hidden row rounded to bf16
    and coded with a2, both saturating -- written with numpy, torch's casts
    and the routing's argmax."""
    cfg = WL.MoEConfig("f8s", M=10, K=256, N=256, E=2, topk=1, seed=27)
    d = WL.make_inputs(cfg)
    N = cfg.N
    q1, s1, q2, s2 = [], [], [], []
    for e in range(2):
        a, b = _rowwise_quant_torch(d["w1"][e].float().numpy())
        c, dd = _rowwise_quant_torch(d["w2"][e].float().numpy())
        q1.append(a); s1.append(b); q2.append(c); s2.append(dd)
    W = orc.Weights(orc.FP8_TENSOR, np.stack(q1), np.stack(q2), np.stack(s1), np.stack(s2))
    ref_ids = np.argmax(d["logits"].numpy(), axis=1)
    x32 = d["x"].float().numpy()
    a1 = np.float32(np.abs(x32).max()) / np.float32(448) * np.float32(0.5)  # saturates x's tail

    def deq(q, s):
        return torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy() * s

    xd = deq(_clamped_cast(x32, a1), float(a1))
    hs = []
    for t in range(cfg.M):
        e = ref_ids[t]
        w1d = deq(q1[e], s1[e].astype(np.float64)[:, None])
        hs.append(_silu(xd[t] @ w1d[:N].T) * (xd[t] @ w1d[N:].T))
    hb = torch.from_numpy(np.stack(hs).astype(np.float32)).to(torch.bfloat16).float().numpy()
    a2 = np.float32(np.abs(hb).max()) / np.float32(448) * np.float32(0.7)  # saturates H's tail
    hq = _clamped_cast(hb, a2)
    assert np.any((hq & 0x7f) == 0x7e)
    hd = deq(hq, float(a2))
    ref = np.stack([hd[t] @ deq(q2[ref_ids[t]], s2[ref_ids[t]].astype(np.float64)[:, None]).T
                    for t in range(cfg.M)])
    out, ids, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1, orc.SOFTMAX,
                                  W, requant_h=True, static_scales=(a1, a2))
    assert np.array_equal(ids[:, 0], ref_ids)
    np.testing.assert_allclose(out, ref, rtol=0, atol=2e-3 * np.abs(ref).max())
    # and not the layer with the tensors' own scales
    dyn, _, _ = orc.moe_forward(_bits(d["x"]), d["logits"].numpy(), None, 1, orc.SOFTMAX,
                                W, requant_h=True)
    assert np.abs(dyn - out).max() > 1e-3 * np.abs(ref).max()
