"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the same
seeded inputs: indices bit-exact, values within the tolerance of the layer's
precision (max|d| <= 2e-2 max|ref| for bf16, 5e-2 for FP8)."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import (TOL, GpuWeights, assert_close_rel, check_ids, gbmoe,
                        oracle_forward, oracle_pair_rows, oracle_weights, run_forward,
                        run_stages)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


# ------------------------------------------------------------------ router --

ROUTE_CFGS = [WL.TINY, WL.SMALL_BF16, WL.SMALL_SIGMOID, WL.MIXTRAL_PREFILL,
              WL.DSV3_PREFILL_FP8, WL.DSV3_DECODE,
              # 262144 tokens: 32768 blocks of the route kernel, 2 M (token, slot) pairs
              WL.MoEConfig("route_M262144_E256_top8_grouped", M=1 << 18, K=128, N=128, E=256,
                           topk=8, score_fn=WL.SIGMOID, n_groups=8, topk_groups=4,
                           zipf_bias=True, seed=64)]


@pytest.mark.parametrize("cfg", ROUTE_CFGS, ids=lambda c: c.name)
def test_route_parity(cfg):
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV, with_weights=False)
    ids = torch.empty((cfg.M, cfg.topk), dtype=torch.int32, device=DEV)
    w = torch.empty((cfg.M, cfg.topk), dtype=torch.float32, device=DEV)
    g.moe_topk_route(d["logits"], d["bias"], cfg.topk, cfg.score_fn, cfg.n_groups,
                     cfg.topk_groups, cfg.renorm, ids, w)
    torch.cuda.synchronize()
    rid, rw, margin = orc.route(d["logits"].cpu().numpy(),
                                None if d["bias"] is None else d["bias"].cpu().numpy(),
                                cfg.topk, cfg.score_fn, cfg.n_groups, cfg.topk_groups,
                                cfg.renorm)
    gid = ids.cpu().numpy()
    diff = check_ids(gid, rid, margin, cfg.name, cfg, d["logits"].cpu().numpy(),
                     None if d["bias"] is None else d["bias"].cpu().numpy())
    same = np.setdiff1d(np.arange(cfg.M), diff)
    np.testing.assert_allclose(w.cpu().numpy()[same], rw[same], atol=2e-6, rtol=0)


def test_route_unrenormalised_and_ungrouped():
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(31)
    for E, k, fn in ((8, 2, orc.SOFTMAX), (256, 8, orc.SIGMOID), (512, 32, orc.SOFTMAX),
                     (40, 3, orc.SIGMOID)):
        lg = torch.randn((257, E), generator=gen, device=DEV)
        lg[:16] = lg[:16].round()  # exact ties
        ids = torch.empty((257, k), dtype=torch.int32, device=DEV)
        w = torch.empty((257, k), dtype=torch.float32, device=DEV)
        g.moe_topk_route(lg, None, k, fn, 1, 1, False, ids, w)
        rid, rw, _ = orc.route(lg.cpu().numpy(), None, k, fn, 1, 1, False)
        assert np.array_equal(ids.cpu().numpy(), rid)
        np.testing.assert_allclose(w.cpu().numpy(), rw, atol=2e-6, rtol=0)


def test_route_grouped_exact_key_ties():
    """Sigmoid grouped routing with logits on a 0.5 grid: many groups share
    their two best values, so their keys tie exactly and the group choice
    falls to the lower group index (keys closer than the fp32 estimate's
    margin are recomputed exactly).  Keys that differ are far apart on this
    grid, so the ids must equal the oracle's on every token."""
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(53)
    for E, n_groups, topk_groups, k in ((64, 8, 4, 6), (256, 8, 4, 8), (32, 4, 2, 3)):
        lg = (torch.randint(-4, 5, (333, E), generator=gen, device=DEV).float() * 0.5)
        ids = torch.empty((333, k), dtype=torch.int32, device=DEV)
        w = torch.empty((333, k), dtype=torch.float32, device=DEV)
        g.moe_topk_route(lg, None, k, orc.SIGMOID, n_groups, topk_groups, True, ids, w)
        rid, rw, _ = orc.route(lg.cpu().numpy(), None, k, orc.SIGMOID, n_groups, topk_groups, True)
        assert np.array_equal(ids.cpu().numpy(), rid), f"E={E}"
        np.testing.assert_allclose(w.cpu().numpy(), rw, atol=2e-6, rtol=0)


# -------------------------------------------------------- count / permute --

@pytest.mark.parametrize("E,M,k,skew", [(8, 64, 2, 0.0), (256, 8192, 8, 1.1),
                                        (32, 1, 1, 0.0), (512, 3001, 5, 2.0),
                                        (256, 1 << 20, 8, 1.1), (512, 99999, 32, 0.5)])
def test_count_and_align_bit_exact(E, M, k, skew):
    """Counts, offsets, sorted pair ids and inv bit-exact against the oracle's
    stable counting sort, up to 8.4 M pairs (4096 sort chunks) and top-32 of
    512 experts."""
    g = gbmoe()
    rng = np.random.default_rng(E * 7 + M)
    p = np.arange(1, E + 1, dtype=np.float64) ** -skew
    ids_np = rng.choice(E, size=(M, k), p=p / p.sum()).astype(np.int32)
    ids = torch.from_numpy(ids_np).to(DEV)
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    counts2 = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    srt = torch.full((M * k,), -5, dtype=torch.int32, device=DEV)
    inv = torch.empty(M * k, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_ALIGN, M, E, 0, 0, k, 0)
    g.moe_count_expert_tokens(ids, E, counts, err)
    g.moe_align_permute(ids, E, counts2, offsets, srt, inv, ws, err)
    rc, bad = orc.count(ids_np, E)
    ro, rs, ri = orc.align(ids_np, E)
    assert bad == 0 and err.item() == 0
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(counts2.cpu().numpy(), rc)
    assert counts.sum().item() == M * k  # every pair lands in one expert
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(srt.cpu().numpy(), rs)
    assert np.array_equal(inv.cpu().numpy(), ri)


def test_align_skips_bad_ids_and_flags_them():
    g = gbmoe()
    E = 6
    ids_np = np.array([[0, 5], [6, 1], [-1, 2], [5, 5]], np.int32)
    ids = torch.from_numpy(ids_np).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    srt = torch.full((8,), -5, dtype=torch.int32, device=DEV)
    inv = torch.empty(8, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    g.moe_align_permute(ids, E, counts, offsets, srt, inv, g.workspace(g.WS_ALIGN, 4, E, 0, 0, 2, 0), err)
    ro, rs, ri = orc.align(ids_np, E)
    assert err.item() & g.ERR_BAD_EXPERT_ID
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(srt.cpu().numpy()[: ro[E]], rs)
    assert np.array_equal(inv.cpu().numpy(), ri)
    assert list(srt.cpu().numpy()[ro[E]:]) == [-5] * (8 - ro[E])


# ------------------------------------------------------------------ quant --

def test_quant_fp8_group_bit_exact():
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(41)
    M, K = 333, 1024
    x = (torch.randn((M, K), generator=gen, device=DEV) *
         torch.logspace(-4, 3, K, device=DEV)).to(torch.bfloat16)
    x[5, :128] = 0
    x[6, 128:256] = -0.0
    x[7, :] = x[7, :].abs() * -1
    q = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    s = torch.empty((M, K // 128), dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_group(x, q, s)
    rq, rs = orc.quant_fp8_group(WL.bf16_bits(x))
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("case", ["all_local", "expert_map", "weight_on_input"])
@pytest.mark.parametrize("mode", ["groups_of_128", "one_scale_per_row", "tensor_dynamic",
                                  "tensor_static"])
def test_quant_fp8_group_permute_bit_exact(case, mode):
    """Quantisation and permutation in one pass (1 x 128 groups, one scale per
    row, or one scale for the tensor, from its maximum or given): codes and
    group-major scales
    of every permuted row bit-exact against the oracle's group quantiser and
    stable sort (A[i] = codes of token sorted[i] / topk), pairs not routed to
    a local expert skipped, rows at and beyond the local total untouched;
    with a row weight (top-1) the product is quantised."""
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(43)
    M, K, E = 300, 640, 16
    topk = 1 if case == "weight_on_input" else 4
    x = (torch.randn((M, K), generator=gen, device=DEV) *
         torch.logspace(-3, 2, K, device=DEV)).to(torch.bfloat16)
    ids = torch.stack([torch.randperm(E, generator=gen, device=DEV)[:topk] for _ in range(M)]).int()
    emap = None
    E_loc = E
    if case == "expert_map":  # experts 4..11 are local (as 0..7), the rest elsewhere
        emap = torch.full((E,), -1, dtype=torch.int32, device=DEV)
        emap[4:12] = torch.arange(8, dtype=torch.int32, device=DEV)
        E_loc = 8
    rw = (torch.rand((M,), generator=gen, device=DEV) + 0.25) if case == "weight_on_input" else None
    P = M * topk
    counts = torch.empty(E_loc, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E_loc + 1, dtype=torch.int32, device=DEV)
    srt = torch.empty(P, dtype=torch.int32, device=DEV)
    inv = torch.empty(P, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_ALIGN, M, E, 0, 0, topk, 0)
    g.moe_align_permute(ids, E_loc, counts, offsets, srt, inv, ws, expert_map=emap,
                        E_global=E if emap is not None else None)
    ld = (P + 3) // 4 * 4
    A = torch.full((P, K), 0xA5, dtype=torch.uint8, device=DEV)
    grouped = mode == "groups_of_128"
    As = torch.full((K // 128 if grouped else 1, ld), -7.0, dtype=torch.float32, device=DEV)
    rwn = None if rw is None else rw.cpu().numpy()
    if grouped:
        g.moe_quant_fp8_group_permute(x, inv, topk, A, As, row_weights=rw)
        rq, rs = orc.quant_fp8_group(WL.bf16_bits(x), group=128, row_weights=rwn)
    elif mode == "one_scale_per_row":  # moe_quant_fp8_row_permute: A_scales[row]
        g.moe_quant_fp8_row_permute(x, inv, topk, A, As.view(-1), row_weights=rw)
        rq, rs = orc.quant_fp8_group(WL.bf16_bits(x), group=K, row_weights=rwn)
    else:  # moe_quant_fp8_tensor_permute: one scale, repeated on every row
        s_static = np.float32(0.02) if mode == "tensor_static" else None
        amax = torch.empty(1, dtype=torch.int32, device=DEV)
        g.moe_quant_fp8_tensor_permute(
            x, inv, topk, A, As.view(-1), amax_ws=amax, row_weights=rw,
            scale=None if s_static is None else torch.tensor([s_static], device=DEV))
        rq, s1 = orc.quant_fp8_tensor(WL.bf16_bits(x), row_weights=rwn, scale=s_static)
        rs = np.full((M, 1), s1, np.float32)
    torch.cuda.synchronize()
    ro, rsrt, rinv = orc.align(ids.cpu().numpy(), E,
                               expert_map=None if emap is None else emap.cpu().numpy(),
                               E_local=E_loc)
    total = int(ro[E_loc])
    assert total == int(offsets[E_loc].item())
    assert np.array_equal(inv.cpu().numpy(), rinv)
    tok = rsrt[:total] // topk
    a = A.cpu().numpy()
    a_s = As.cpu().numpy()
    assert np.array_equal(a[:total], rq[tok])
    assert np.array_equal(a_s[:, :total], rs[tok].T)
    assert np.all(a[total:] == 0xA5) and np.all(a_s[:, total:] == -7.0)


@pytest.mark.parametrize("K,weighted", [(1024, False), (7168, True), (640, False)])
def test_quant_fp8_rowwise_bit_exact(K, weighted):
    """One scale per row (per-token activations, per-channel weights): codes
    and scales bit-exact against the oracle, with and without row weights."""
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(43 + K)
    M = 301
    x = (torch.randn((M, K), generator=gen, device=DEV) *
         torch.logspace(-3, 2, K, device=DEV)).to(torch.bfloat16)
    x[5] = 0
    x[7] = x[7].abs() * -1
    rw = (torch.rand(M, generator=gen, device=DEV) + 0.05) if weighted else None
    q = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    s = torch.empty((M, 1), dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_group(x, q, s, group=K, row_weights=rw)
    rq, rs = orc.quant_fp8_group(WL.bf16_bits(x), group=K,
                                 row_weights=None if rw is None else rw.cpu().numpy())
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("weighted,partial", [(False, False), (True, False), (False, True)])
def test_quant_fp8_tensor_bit_exact(weighted, partial):
    """One scale for the whole tensor: the scale, every code and every row's
    copy of the scale bit-exact; with a device row count only the first rows
    count and the rest are left as they were."""
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(47)
    M, K = 333, 1024
    x = (torch.randn((M, K), generator=gen, device=DEV) *
         torch.logspace(-2, 1, M, device=DEV)[:, None]).to(torch.bfloat16)
    rw = (torch.rand(M, generator=gen, device=DEV) + 0.05) if weighted else None
    n = 200 if partial else M
    n_rows = torch.tensor([n], dtype=torch.int32, device=DEV) if partial else None
    q = torch.full((M, K), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    amax = torch.empty(1, dtype=torch.int32, device=DEV)
    g.moe_quant_fp8_tensor(x, q, s, amax, n_rows=n_rows, row_weights=rw)
    rq, rs = orc.quant_fp8_tensor(WL.bf16_bits(x[:n]),
                                  row_weights=None if rw is None else rw[:n].cpu().numpy())
    assert np.all(s[:n].cpu().numpy() == rs)
    assert np.array_equal(q[:n].cpu().numpy(), rq)
    assert torch.all(q[n:] == 0xAB) and torch.all(s[n:] == -1.0)


@pytest.mark.parametrize("cfg", [WL.SMALL_FP8T, WL.MID_FP8T], ids=lambda c: c.name)
def test_forward_parity_fp8_tensor(cfg):
    """Per-tensor activation scales: every token against the oracle's
    two-pass layer (the scales of x and H span all tokens)."""
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    out, ids, wts, err = run_forward(cfg, d, gw)
    torch.cuda.synchronize()
    assert err.item() == 0
    W = oracle_weights(cfg, d["w1"], d["w2"])
    ref, rid, rw = oracle_forward(cfg, d, W)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[cfg.dtype], cfg.name)


@pytest.mark.parametrize("partial", [False, True], ids=["all_rows", "device_row_count"])
def test_quant_fp8_tensor_static_bit_exact(partial):
    """A static per-tensor scale (the quant config's a1_scale): every code of
    x / scale bit-exact with the oracle's, the largest values saturated at
    +-448, the scale copied to every counted row, the other rows untouched."""
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(48)
    M, K = 333, 1024
    x = (torch.randn((M, K), generator=gen, device=DEV) *
         torch.logspace(-2, 1, M, device=DEV)[:, None]).to(torch.bfloat16)
    rw = torch.rand(M, generator=gen, device=DEV) + 0.05
    n = 200 if partial else M
    n_rows = torch.tensor([n], dtype=torch.int32, device=DEV) if partial else None
    v = (x[:n].float() * rw[:n, None]).abs().max().item()  # the counted rows' largest |x w|
    s_host = np.float32(v) / np.float32(448) * np.float32(0.3)
    scale = torch.tensor([s_host], dtype=torch.float32, device=DEV)
    q = torch.full((M, K), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_tensor_static(x, scale, q, s, n_rows=n_rows, row_weights=rw)
    rq, rs = orc.quant_fp8_tensor(WL.bf16_bits(x[:n]), row_weights=rw[:n].cpu().numpy(),
                                  scale=s_host)
    assert np.all(s[:n].cpu().numpy() == rs)
    assert np.array_equal(q[:n].cpu().numpy(), rq)
    assert np.any((rq & 0x7f) == 0x7e)  # saturated codes among them
    assert torch.all(q[n:] == 0xAB) and torch.all(s[n:] == -1.0)


@pytest.mark.parametrize("cfg", [WL.SMALL_FP8T, WL.MID_FP8T], ids=lambda c: c.name)
def test_forward_parity_fp8_tensor_static_scales(cfg):
    """Static per-tensor activation scales a1 (x) and a2 (H), small enough
    that both saturate their largest values: every token against the
    oracle's layer with the same scales; chunked equals unchunked bit for
    bit (no scale depends on the chunk)."""
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    a1 = np.float32(d["x"].float().abs().max().item()) / np.float32(448) * np.float32(0.5)
    a2 = np.float32(0.01)
    a1_t = torch.tensor([a1], dtype=torch.float32, device=DEV)
    a2_t = torch.tensor([a2], dtype=torch.float32, device=DEV)
    out, ids, wts, err = run_forward(cfg, d, gw, a1_scale=a1_t, a2_scale=a2_t)
    torch.cuda.synchronize()
    assert err.item() == 0
    W = oracle_weights(cfg, d["w1"], d["w2"])
    ref, rid, rw = oracle_forward(cfg, d, W, static_scales=(a1, a2))
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[cfg.dtype], cfg.name + " static")
    dyn, _, _, _ = run_forward(cfg, d, gw)
    assert not torch.equal(dyn.view(torch.int16), out.view(torch.int16))
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    chunk = 100
    outc = torch.empty_like(out)
    g.moe_forward_chunked(d["x"], d["logits"], d["bias"], N, E, k, cfg.score_fn, cfg.n_groups,
                          cfg.topk_groups, cfg.renorm, cfg.dtype, gw.w1, gw.w1s, gw.w2, gw.w2s,
                          outc, g.workspace(g.WS_FORWARD, chunk, E, N, K, k, cfg.dtype), chunk,
                          a1_scale=a1_t, a2_scale=a2_t)
    torch.cuda.synchronize()
    assert torch.equal(outc.view(torch.int16), out.view(torch.int16))


def test_quant_fp8_block_bit_exact():
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(42)
    w = (torch.randn((3, 256, 384), generator=gen, device=DEV) * 0.03).to(torch.bfloat16)
    q = torch.empty(w.shape, dtype=torch.uint8, device=DEV)
    s = torch.empty((3, 2, 3), dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_block(w, q, s)
    for e in range(3):
        rq, rs = orc.quant_fp8_block(WL.bf16_bits(w[e]))
        assert np.array_equal(s[e].cpu().numpy(), rs)
        assert np.array_equal(q[e].cpu().numpy(), rq)


# ------------------------------------------------------- expert GEMMs ------

def _stage_inputs(cfg):
    """Route with the oracle (inputs for the GEMM stages never come from the
    CUDA path), then permute on the GPU."""
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    rid, rw, _ = orc.route(d["logits"].cpu().numpy(),
                           None if d["bias"] is None else d["bias"].cpu().numpy(),
                           cfg.topk, cfg.score_fn, cfg.n_groups, cfg.topk_groups,
                           cfg.renorm)
    ids = torch.from_numpy(rid).to(DEV)
    wts = torch.from_numpy(rw.astype(np.float32)).to(DEV)
    P = cfg.P
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device=DEV)
    srt = torch.empty(P, dtype=torch.int32, device=DEV)
    inv = torch.empty(P, dtype=torch.int32, device=DEV)
    g.moe_align_permute(ids, cfg.E, None, offsets, srt, inv,
                        g.workspace(g.WS_ALIGN, cfg.M, cfg.E, 0, 0, cfg.topk, 0))
    return d, rid, rw, ids, wts, offsets, srt, inv


SMALL_STANDARD = [WL.TINY, WL.SMALL_BF16, WL.SMALL_SIGMOID, WL.SMALL_FP8, WL.SMALL_PAIR,
                  WL.SMALL_PAIR_TOP2, WL.SMALL_FP8_K640, WL.SMALL_FP8_NARROW, WL.SMALL_FP8CH,
                  WL.SMALL_FP8CH_PAIR]


@pytest.mark.parametrize("cfg", SMALL_STANDARD, ids=lambda c: c.name)
def test_gate_up_then_down_stages(cfg):
    """Each grouped GEMM against the oracle's expert rows."""
    g = gbmoe()
    d, rid, rw, ids, wts, offsets, srt, inv = _stage_inputs(cfg)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    W = oracle_weights(cfg, d["w1"], d["w2"])
    M, E, N, K, k, P = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk, cfg.P
    fp8 = cfg.dtype == WL.FP8
    ch = cfg.dtype == WL.FP8_CHANNEL
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if ch:  # one scale per token; H in bf16, then one scale per row of H
        xq = torch.empty((M, K), dtype=torch.uint8, device=DEV)
        xs = torch.empty((M, 1), dtype=torch.float32, device=DEV)
        g.moe_quant_fp8_group(d["x"], xq, xs, group=K)
        xin, xin_s = xq, xs
        H = torch.empty((P, N), dtype=torch.bfloat16, device=DEV)
        Hs = None
    elif fp8:
        xq = torch.empty((M, K), dtype=torch.uint8, device=DEV)
        xs = torch.empty((M, K // 128), dtype=torch.float32, device=DEV)
        g.moe_quant_fp8_group(d["x"], xq, xs)
        xin, xin_s = xq, xs
        H = torch.empty((P, N), dtype=torch.uint8, device=DEV)
        ld = (P + 3) // 4 * 4  # group-major scales, leading dimension rounded to 4
        Hs = torch.empty((N // 128, ld), dtype=torch.float32, device=DEV)
    else:
        xin, xin_s = d["x"], None
        H = torch.empty((P, N), dtype=torch.bfloat16, device=DEV)
        Hs = None
    A = torch.empty((P, K), dtype=xin.dtype, device=DEV)
    ld = (P + 3) // 4 * 4
    As = (torch.empty((K // 128, ld), dtype=torch.float32, device=DEV) if fp8 else
          torch.empty((1, ld), dtype=torch.float32, device=DEV) if ch else None)
    g.moe_permute_rows(xin, xin_s, srt, offsets, k, E, cfg.dtype, A, As)
    g.moe_grouped_gemm_gate_up_silu(A, As, offsets, M, k, E, N, K, gw.w1, gw.w1s,
                                    cfg.dtype, H, Hs, err)
    y = torch.empty((M, k, K), dtype=torch.bfloat16, device=DEV)
    Hd, Hds = H, Hs
    if ch:
        Hd = torch.empty((P, N), dtype=torch.uint8, device=DEV)
        Hds = torch.empty((P, 1), dtype=torch.float32, device=DEV)
        g.moe_quant_fp8_group(H, Hd, Hds, group=N)
    g.moe_grouped_gemm_down(Hd, Hds, srt, offsets, wts, M, k, E, N, K, gw.w2, gw.w2s,
                            cfg.dtype, y, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    if fp8:
        Hf = (H.view(torch.float8_e4m3fn).float().view(P, N // 128, 128) *
              Hs[:, :P].t().reshape(P, N // 128, 1)).view(P, N).cpu().numpy()
    elif ch:  # the codes the down GEMM read, dequantised
        Hf = (Hd.view(torch.float8_e4m3fn).float() * Hds).cpu().numpy()
    else:
        Hf = H.float().cpu().numpy()
    yf = y.float().cpu().numpy()
    srt_np = srt.cpu().numpy()
    xbits = WL.bf16_bits(d["x"])
    rows = range(P) if P <= 600 else np.random.default_rng(0).choice(P, 600, replace=False)
    href = np.zeros((len(rows), N))
    yref = np.zeros((len(rows), K))
    hgot = np.zeros_like(href)
    ygot = np.zeros_like(yref)
    for n, i in enumerate(rows):
        pair = srt_np[i]
        t, j = divmod(int(pair), k)
        h, yy = orc.expert_row(xbits, t, rid[t, j], W, requant_h=cfg.requant_h)
        href[n] = h
        yref[n] = rw[t, j] * yy
        hgot[n] = Hf[i]
        ygot[n] = yf[t, j]
    assert_close_rel(hgot, href, TOL[cfg.dtype], "H")
    assert_close_rel(ygot, yref, TOL[cfg.dtype], "weighted y")


@pytest.mark.parametrize("cfg", SMALL_STANDARD, ids=lambda c: c.name)
def test_forward_parity_small(cfg):
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    out, ids, wts, err = run_forward(cfg, d, gw)
    torch.cuda.synchronize()
    assert err.item() == 0
    W = oracle_weights(cfg, d["w1"], d["w2"])
    ref, rid, rw = oracle_forward(cfg, d, W)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, atol=2e-6, rtol=0)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[cfg.dtype], cfg.name)


@pytest.mark.parametrize("cfg,static", [(WL.SMALL_FP8T, False), (WL.SMALL_FP8T, True),
                                        (WL.SMALL_FP8CH, False), (WL.SMALL_FP8, False)],
                         ids=["fp8_tensor_dynamic", "fp8_tensor_static", "fp8_channel",
                              "fp8_block"])
def test_forward_equals_its_separate_calls(cfg, static):
    """The one-call layer (which quantises and permutes x in one pass) equals
    the same layer run as its separate calls (quantise, then gather) bit for
    bit, on every token; per-tensor e4m3 with dynamic and with static
    activation scales."""
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    kw = {}
    if static:
        a1 = np.float32(d["x"].float().abs().max().item()) / np.float32(448) * np.float32(0.5)
        kw = dict(a1_scale=torch.tensor([a1], dtype=torch.float32, device=DEV),
                  a2_scale=torch.tensor([0.01], dtype=torch.float32, device=DEV))
    out, ids, wts, err = run_forward(cfg, d, gw, **kw)
    st = run_stages(cfg, d, gw, ids, wts, **kw)
    torch.cuda.synchronize()
    assert err.item() == 0 and st["err"].item() == 0
    assert torch.equal(out.view(torch.int16), st["out"].view(torch.int16))


def test_forward_is_deterministic():
    cfg = WL.SMALL_SIGMOID
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    a, _, _, _ = run_forward(cfg, d, gw)
    b, _, _, _ = run_forward(cfg, d, gw)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M", [0, 1, 129])
def test_forward_edge_sizes(M):
    """Empty input is a no-op; one token and a 129-token ragged tail."""
    base = WL.SMALL_BF16
    cfg = WL.MoEConfig("edge", M=M, K=base.K, N=base.N, E=base.E, topk=base.topk, seed=5)
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    if M == 0:
        g = gbmoe()
        out = torch.full((1, cfg.K), 3.0, dtype=torch.bfloat16, device=DEV)
        ws = torch.empty(256, dtype=torch.uint8, device=DEV)
        g.moe_forward(d["x"], d["logits"], None, cfg.N, cfg.E, cfg.topk, cfg.score_fn,
                      1, 1, True, cfg.dtype, gw.w1, None, gw.w2, None, out, ws)
        torch.cuda.synchronize()
        assert torch.all(out == 3.0)
        return
    out, _, _, err = run_forward(cfg, d, gw)
    torch.cuda.synchronize()
    W = oracle_weights(cfg, d["w1"], d["w2"])
    ref, _, _ = oracle_forward(cfg, d, W)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[cfg.dtype], f"M={M}")


@pytest.mark.parametrize("M", [300, 600])
def test_one_expert_takes_every_token_matches_torch_matmul(M):
    """All tokens on one expert: the grouped GEMMs reduce to dense matmuls,
    checked against torch's own bf16 matmul on the GPU (a second reference).
    M = 600 over 4 experts runs on CTA pairs (two full 256-row tiles and a
    tail of 88), M = 300 on the 1-SM kernel."""
    g = gbmoe()
    cfg = WL.MoEConfig("one", M=M, K=512, N=256, E=4, topk=1, seed=6)
    d = WL.make_inputs(cfg, DEV)
    d["logits"][:, 2] += 100.0  # every token picks expert 2
    out, ids, wts, err = run_forward(cfg, d, GpuWeights(cfg, d["w1"], d["w2"]))
    torch.cuda.synchronize()
    assert torch.all(ids == 2)
    x = d["x"].float()
    w1 = d["w1"][2].float()
    h = torch.nn.functional.silu(x @ w1[:256].T) * (x @ w1[256:].T)
    ref = (h.to(torch.bfloat16).float() @ d["w2"][2].float().T)
    assert_close_rel(out.float().cpu().numpy(), ref.cpu().numpy(), 2e-2, "dense")


# ------------------------------------------------------------- full-size ---

FULL_CFGS = [WL.MIXTRAL_PREFILL, WL.DSV3_DECODE, WL.DSV3_PREFILL_FP8, WL.DSV3_PREFILL_FP8CH]
N_SAMPLE = 512


@pytest.mark.parametrize("cfg", FULL_CFGS, ids=lambda c: c.name)
def test_forward_parity_full_size(cfg):
    """The bench's workloads at full size, checked as follows (tokens are
    independent, so every checked row is computed exactly as in the full
    run):
      * routing: the ids of every token bit for bit (a near-tie token must be
        one of the valid choices), the weights of the others;
      * counts, offsets, sorted pair ids and inv of the workload's own routing
        (the oracle's ids, aligned on the GPU) bit for bit;
      * the weighted expert row of every pair routed to the two most loaded
        experts (the heavy experts' tiles), against the oracle;
      * the output of a seeded sample of 512 tokens (every token when there
        are fewer), against the oracle's layer;
      * the one-call layer bit for bit equal, on every token, to the same
        layer run as its separate calls on the same routing."""
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    out, ids, wts, err = run_forward(cfg, d, gw)
    torch.cuda.synchronize()
    assert err.item() == 0
    lg = d["logits"].cpu().numpy()
    bias = None if d["bias"] is None else d["bias"].cpu().numpy()
    rid, rw, margin = orc.route(lg, bias, cfg.topk, cfg.score_fn, cfg.n_groups,
                                cfg.topk_groups, cfg.renorm)
    gid = ids.cpu().numpy()
    diff = check_ids(gid, rid, margin, cfg.name, cfg, lg, bias)
    same = np.setdiff1d(np.arange(cfg.M), diff)
    np.testing.assert_allclose(wts.cpu().numpy()[same], rw[same], atol=2e-6, rtol=0)

    # the permutation of the workload's routing, every pair
    E, P = cfg.E, cfg.P
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    srt = torch.full((P,), -5, dtype=torch.int32, device=DEV)
    inv = torch.empty(P, dtype=torch.int32, device=DEV)
    aerr = torch.zeros(1, dtype=torch.int32, device=DEV)
    g.moe_align_permute(torch.from_numpy(rid).to(DEV), E, counts, offsets, srt, inv,
                        g.workspace(g.WS_ALIGN, cfg.M, E, 0, 0, cfg.topk, 0), aerr)
    rc, bad = orc.count(rid, E)
    ro, rs, ri = orc.align(rid, E)
    torch.cuda.synchronize()
    assert bad == 0 and aerr.item() == 0 and rc.sum() == P
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(srt.cpu().numpy(), rs)
    assert np.array_equal(inv.cpu().numpy(), ri)
    del counts, offsets, srt, inv

    # the layer as separate calls on the path's own routing
    st = run_stages(cfg, d, gw, ids, wts)
    torch.cuda.synchronize()
    assert st["err"].item() == 0
    assert torch.equal(out.view(torch.int16), st["out"].view(torch.int16)), \
        "one-call layer differs from its separate calls"

    # every pair of the two most loaded experts (tokens with a near-tie route
    # left out: their experts differ from the oracle's)
    top2 = np.argsort(-rc, kind="stable")[:2]
    pairs = np.concatenate([rs[ro[e]:ro[e + 1]] for e in top2])
    pairs = pairs[~np.isin(pairs // cfg.topk, diff)]
    yref = oracle_pair_rows(cfg, d, d["w1"], d["w2"], rid, pairs) * rw.ravel()[pairs][:, None]
    ygot = st["y_slot"].view(P, cfg.K)[torch.from_numpy(pairs).to(DEV)].float().cpu().numpy()
    assert_close_rel(ygot, yref, TOL[cfg.dtype], f"{cfg.name}: pairs of experts {top2}")
    del st

    # a seeded sample of tokens through the whole layer
    rng = np.random.default_rng(1)
    tokens = (np.arange(cfg.M) if cfg.M <= N_SAMPLE
              else np.sort(rng.choice(cfg.M, N_SAMPLE, replace=False)))
    tokens = np.setdiff1d(tokens, diff)
    W = oracle_weights(cfg, d["w1"], d["w2"], np.unique(rid[tokens]))
    ref, rid_s, _ = oracle_forward(cfg, d, W, tokens=tokens)
    assert np.array_equal(rid_s, rid[tokens])
    assert_close_rel(out[torch.from_numpy(tokens).to(DEV)].float().cpu().numpy(), ref,
                     TOL[cfg.dtype], cfg.name)


def test_forward_parity_fp8_tensor_static_full_size_sampled():
    """The DeepSeek-V3-shaped prefill with per-tensor e4m3 activations and
    static scales for x and H (small enough that both saturate their largest
    values) at full size: the ids and outputs of a seeded sample of 512
    tokens against the oracle's layer with the same scales (no scale depends
    on other tokens, so the sampled tokens are computed exactly as in the
    full run)."""
    cfg = WL.DSV3_PREFILL_FP8T
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    a1 = np.float32(d["x"].float().abs().max().item()) / np.float32(448) * np.float32(0.8)
    a2 = np.float32(0.03)
    out, ids, wts, err = run_forward(
        cfg, d, gw, a1_scale=torch.tensor([a1], dtype=torch.float32, device=DEV),
        a2_scale=torch.tensor([a2], dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    assert err.item() == 0
    lg = d["logits"].cpu().numpy()
    bias = None if d["bias"] is None else d["bias"].cpu().numpy()
    rid, _, margin = orc.route(lg, bias, cfg.topk, cfg.score_fn, cfg.n_groups,
                               cfg.topk_groups, cfg.renorm)
    diff = check_ids(ids.cpu().numpy(), rid, margin, cfg.name, cfg, lg, bias)
    rng = np.random.default_rng(2)
    tokens = np.setdiff1d(np.sort(rng.choice(cfg.M, N_SAMPLE, replace=False)), diff)
    W = oracle_weights(cfg, d["w1"], d["w2"], np.unique(rid[tokens]))
    ref, rid_s, _ = oracle_forward(cfg, d, W, tokens=tokens, static_scales=(a1, a2))
    assert np.array_equal(rid_s, rid[tokens])
    assert_close_rel(out[torch.from_numpy(tokens).to(DEV)].float().cpu().numpy(), ref,
                     TOL[cfg.dtype], cfg.name + " static scales")


def test_forward_parity_fp8_tensor_dynamic_full_size():
    """The DeepSeek-V3-shaped prefill with per-tensor e4m3 activations and
    dynamic scales, at full size.  The scale of H spans all 65536 hidden rows,
    more than the oracle computes here, so the check is a chain:
    - x's scale and codes equal the oracle's quantiser, bit for bit;
    - H's scale is the maximum magnitude of the hidden rows the gate/up GEMM
      wrote (over the computed rows only) / 448, and H's codes are torch's
      saturating e4m3 cast of those rows divided by it;
    - the one-call layer equals its separate calls, and equals the layer run
      with those two scales given as static scales, bit for bit (the static
      path at full size is checked against the oracle in the test above)."""
    cfg = WL.DSV3_PREFILL_FP8T
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    out, ids, wts, err = run_forward(cfg, d, gw)
    torch.cuda.synchronize()
    assert err.item() == 0
    st = run_stages(cfg, d, gw, ids, wts, keep_hidden=True)
    torch.cuda.synchronize()
    assert st["err"].item() == 0
    assert torch.equal(st["out"].view(torch.int16), out.view(torch.int16))
    # x: the oracle's per-tensor quantiser
    q_ref, s_ref = orc.quant_fp8_tensor(WL.bf16_bits(d["x"]))
    xs = st["xs"].view(-1)
    assert torch.all(xs == xs[0])
    assert np.float32(xs[0].item()) == s_ref
    assert np.array_equal(st["xq"].cpu().numpy(), q_ref)
    # H: the maximum of the computed rows, then the saturating cast
    P = int(st["offsets"][cfg.E].item())
    assert P == cfg.M * cfg.topk
    hb = st["Hb"][:P].float().cpu().numpy()  # bf16 values, exact in fp32
    hmax = np.float32(np.abs(hb).max())
    assert np.float32(st["amax"][1:2].view(torch.float32).item()) == hmax
    hs = st["Hs"].view(-1)[:P]
    assert torch.all(hs == hs[0])
    s_h = np.float32(hs[0].item())
    assert s_h == hmax / np.float32(448)  # IEEE fp32 division
    q = np.clip(hb / s_h, np.float32(-448), np.float32(448))
    codes = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(st["H"][:P].cpu().numpy(), codes)
    del hb, q, codes
    # the dynamic layer is the static layer with its own scales
    out_s, _, _, err_s = run_forward(cfg, d, gw, a1_scale=xs[:1].clone(),
                                     a2_scale=hs[:1].clone())
    torch.cuda.synchronize()
    assert err_s.item() == 0
    assert torch.equal(out_s.view(torch.int16), out.view(torch.int16))
