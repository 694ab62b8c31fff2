"""BatchedExperts (E, T, K) masked by device-resident counts: parity with the
oracle, padded rows never read or written, capture in a CUDA graph and
replay with fresh inputs and counts (no host count read)."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import TOL, GpuWeights, assert_close_rel, gbmoe, oracle_weights

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = 0x7E7E  # a bf16 bit pattern no expert output takes by accident


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


def _run(cfg, xb, counts, w1, w2, yb, ws, err, stream=None):
    gbmoe().moe_batched_masked_experts(xb, counts, cfg.N, w1, w2, yb, ws,
                                       err_word=err, stream=stream)


def _fresh(cfg):
    E, T, K = cfg.E, cfg.M, cfg.K
    yb = torch.empty((E, T, K), dtype=torch.bfloat16, device=DEV)
    yb.view(torch.int16).fill_(SENTINEL)
    return yb


def _check_rows(cfg, d, yb, W, rows=None):
    counts = d["counts"].cpu().numpy()
    # e4m3: h requantised per row and 128-group before the down projection
    ref, n = orc.batched_experts(WL.bf16_bits(d["x_b"]), counts, W, rows=rows,
                                 requant_h=cfg.dtype == WL.FP8)
    got = yb.float().cpu().numpy()
    mask = ~np.isnan(ref[..., 0])
    assert mask.sum() == n
    assert_close_rel(got[mask], ref[mask], TOL[cfg.dtype], cfg.name)
    bits = yb.view(torch.int16).cpu().numpy()
    for e in range(cfg.E):
        c = min(max(int(counts[e]), 0), cfg.M)
        assert np.all(bits[e, c:] == np.int16(SENTINEL)), f"padded rows of expert {e} written"


@pytest.mark.parametrize("cfg", [WL.SMALL_BATCHED, WL.SMALL_BATCHED_SHORT],
                         ids=lambda c: c.name)
def test_batched_small_all_rows(cfg):
    d = WL.make_inputs(cfg, DEV)
    g = gbmoe()
    yb = _fresh(cfg)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, WL.BF16)
    _run(cfg, d["x_b"], d["counts"], d["w1"], d["w2"], yb, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    _check_rows(cfg, d, yb, oracle_weights(cfg, d["w1"], d["w2"]))


def test_batched_padding_garbage_does_not_matter():
    cfg = WL.SMALL_BATCHED
    d = WL.make_inputs(cfg, DEV)
    g = gbmoe()
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, WL.BF16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    a = _fresh(cfg)
    _run(cfg, d["x_b"], d["counts"], d["w1"], d["w2"], a, ws, err)
    xb2 = d["x_b"].clone()
    gen = torch.Generator(device=DEV).manual_seed(99)
    for e in range(cfg.E):
        c = int(d["counts"][e])
        xb2[e, c:] = (torch.randn((cfg.M - c, cfg.K), generator=gen, device=DEV) * 1e4).to(torch.bfloat16)
    b = _fresh(cfg)
    _run(cfg, xb2, d["counts"], d["w1"], d["w2"], b, ws, err)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_batched_count_out_of_range_is_clamped_and_flagged():
    cfg = WL.SMALL_BATCHED
    d = WL.make_inputs(cfg, DEV)
    g = gbmoe()
    counts = d["counts"].clone()
    counts[0] = cfg.M + 50
    counts[1] = -3
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, WL.BF16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    yb = _fresh(cfg)
    _run(cfg, d["x_b"], counts, d["w1"], d["w2"], yb, ws, err)
    torch.cuda.synchronize()
    assert err.item() & g.ERR_COUNT_RANGE
    d2 = dict(d)
    d2["counts"] = counts
    _check_rows(cfg, d2, yb, oracle_weights(cfg, d["w1"], d["w2"]))


def test_batched_full_size_graph_replays():
    """E=32, T=1024, K=7168, N=2048: captured once, replayed 50 times with
    fresh seeds copied into the static buffers (inputs and device counts).
    Every replay equals the eager call bit for bit and leaves every padded
    row untouched; every tenth replay (5 of them) also matches the oracle on
    sampled rows of every expert with rows, among them the first and last
    valid row."""
    cfg = WL.BATCHED_MASKED
    g = gbmoe()
    d0 = WL.make_inputs(cfg, DEV, seed=cfg.seed)
    w1, w2 = d0["w1"], d0["w2"]
    xb = d0["x_b"].clone()
    counts = d0["counts"].clone()
    yb = _fresh(cfg)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, WL.BF16)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(cfg, xb, counts, w1, w2, yb, ws, err, stream=s)  # warm up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run(cfg, xb, counts, w1, w2, yb, ws, err)
    rng = np.random.default_rng(7)
    rows_t = torch.arange(cfg.M, device=DEV).view(1, cfg.M)
    eager = _fresh(cfg)
    checked = 0
    for r in range(50):
        dr = WL.make_inputs(cfg, DEV, seed=cfg.seed + r + 1, with_weights=False)
        xb.copy_(dr["x_b"])
        counts.copy_(dr["counts"])
        yb.view(torch.int16).fill_(SENTINEL)
        graph.replay()
        eager.view(torch.int16).fill_(SENTINEL)
        _run(cfg, dr["x_b"], dr["counts"], w1, w2, eager, ws, err)
        torch.cuda.synchronize()
        assert err.item() == 0, f"replay {r}"
        assert torch.equal(eager.view(torch.int16), yb.view(torch.int16)), f"replay {r}"
        pad = rows_t >= dr["counts"].view(cfg.E, 1)
        assert torch.all(yb.view(torch.int16)[pad] == SENTINEL), f"replay {r}: padding written"
        if r % 10 == 0:
            c = dr["counts"].cpu().numpy()
            rows = []
            for e in range(cfg.E):
                if c[e] > 0:
                    pick = {0, int(c[e]) - 1} | set(int(v) for v in rng.choice(c[e], min(2, c[e]),
                                                                          replace=False))
                    rows += [(e, rr) for rr in sorted(pick)]
            rows = np.array(rows, np.int32)
            W = oracle_weights(cfg, w1, w2, np.unique(rows[:, 0]))
            _check_rows(cfg, {"x_b": dr["x_b"], "counts": dr["counts"]}, yb, W, rows=rows)
            checked += 1
    assert checked == 5


# ------------------------------------------------------------------ e4m3 ----

def _quant_xb(xb):
    """x_b (E, T, K) bf16 -> e4m3 codes (E, T, K) and scales (E*T, K/128), by
    the library's group quantiser on the (E*T, K) view (bit-exact with the
    oracle's, which the oracle's own batched path applies to each row)."""
    E, T, K = xb.shape
    q = torch.empty((E, T, K), dtype=torch.uint8, device=xb.device)
    sc = torch.empty((E * T, K // 128), dtype=torch.float32, device=xb.device)
    gbmoe().moe_quant_fp8_group(xb.reshape(E * T, K), q.view(E * T, K), sc)
    return q, sc


def _run_fp8(cfg, q, sc, counts, gw, yb, ws, err, stream=None):
    gbmoe().moe_batched_masked_experts(q, counts, cfg.N, gw.w1, gw.w2, yb, ws, dtype=WL.FP8,
                                       x_b_scales=sc, w1_scales=gw.w1s, w2_scales=gw.w2s,
                                       err_word=err, stream=stream)


@pytest.mark.parametrize("cfg", [WL.SMALL_BATCHED_FP8, WL.SMALL_BATCHED_FP8_K640],
                         ids=lambda c: c.name)
def test_batched_fp8_small_all_rows(cfg):
    """Every valid row against the oracle's e4m3 experts (h requantised);
    padded rows never written."""
    d = WL.make_inputs(cfg, DEV)
    g = gbmoe()
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    q, sc = _quant_xb(d["x_b"])
    yb = _fresh(cfg)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, WL.FP8)
    _run_fp8(cfg, q, sc, d["counts"], gw, yb, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    _check_rows(cfg, d, yb, oracle_weights(cfg, d["w1"], d["w2"]))


def test_batched_fp8_padding_garbage_does_not_matter():
    """Codes and scales of padded rows (here huge, infinite or NaN scales)
    change nothing."""
    cfg = WL.SMALL_BATCHED_FP8
    d = WL.make_inputs(cfg, DEV)
    g = gbmoe()
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    q, sc = _quant_xb(d["x_b"])
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, WL.FP8)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    a = _fresh(cfg)
    _run_fp8(cfg, q, sc, d["counts"], gw, a, ws, err)
    q2, sc2 = q.clone(), sc.clone().view(cfg.E, cfg.M, -1)
    gen = torch.Generator(device=DEV).manual_seed(98)
    for e in range(cfg.E):
        c = int(d["counts"][e])
        q2[e, c:] = torch.randint(0, 256, (cfg.M - c, cfg.K), generator=gen, device=DEV,
                                  dtype=torch.int32).to(torch.uint8)
        sc2[e, c:] = float("nan") if e % 2 else float("inf")
    b = _fresh(cfg)
    _run_fp8(cfg, q2, sc2.view(cfg.E * cfg.M, -1), d["counts"], gw, b, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_batched_fp8_count_out_of_range_is_clamped_and_flagged():
    cfg = WL.SMALL_BATCHED_FP8_K640
    d = WL.make_inputs(cfg, DEV)
    g = gbmoe()
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    q, sc = _quant_xb(d["x_b"])
    counts = d["counts"].clone()
    counts[0] = cfg.M + 7
    counts[1] = -1
    ws = g.workspace(g.WS_BATCHED, cfg.M, cfg.E, cfg.N, cfg.K, 1, WL.FP8)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    yb = _fresh(cfg)
    _run_fp8(cfg, q, sc, counts, gw, yb, ws, err)
    torch.cuda.synchronize()
    assert err.item() & g.ERR_COUNT_RANGE
    d2 = dict(d)
    d2["counts"] = counts
    _check_rows(cfg, d2, yb, oracle_weights(cfg, d["w1"], d["w2"]))


def test_batched_fp8_full_size_graph_replays():
    """E=32, T=1024, K=7168, N=2048 with e4m3 activations and block-scaled
    weights: captured once (quantisation of x_b included), replayed 20 times
    with fresh inputs and counts; every replay equals the eager calls bit for
    bit and leaves the padding untouched; every fifth also matches the oracle
    on sampled rows of every expert with rows (first and last valid row
    among them)."""
    cfg = WL.BATCHED_MASKED_FP8
    g = gbmoe()
    d0 = WL.make_inputs(cfg, DEV, seed=cfg.seed)
    w1, w2 = d0["w1"], d0["w2"]
    gw = GpuWeights(cfg, w1, w2)
    xb = d0["x_b"].clone()
    counts = d0["counts"].clone()
    E, T, K = cfg.E, cfg.M, cfg.K
    q = torch.empty((E, T, K), dtype=torch.uint8, device=DEV)
    sc = torch.empty((E * T, K // 128), dtype=torch.float32, device=DEV)
    yb = _fresh(cfg)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_BATCHED, T, E, cfg.N, K, 1, WL.FP8)

    def layer(out, x, c, stream=None):
        g.moe_quant_fp8_group(x.reshape(E * T, K), q.view(E * T, K), sc, stream=stream)
        _run_fp8(cfg, q, sc, c, gw, out, ws, err, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(yb, xb, counts, stream=s)  # warm up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(yb, xb, counts)
    rng = np.random.default_rng(8)
    rows_t = torch.arange(T, device=DEV).view(1, T)
    eager = _fresh(cfg)
    checked = 0
    for r in range(20):
        dr = WL.make_inputs(cfg, DEV, seed=cfg.seed + r + 1, with_weights=False)
        xb.copy_(dr["x_b"])
        counts.copy_(dr["counts"])
        yb.view(torch.int16).fill_(SENTINEL)
        graph.replay()
        torch.cuda.synchronize()
        got = yb.clone()
        eager.view(torch.int16).fill_(SENTINEL)
        layer(eager, dr["x_b"], dr["counts"])
        torch.cuda.synchronize()
        assert err.item() == 0, f"replay {r}"
        assert torch.equal(eager.view(torch.int16), got.view(torch.int16)), f"replay {r}"
        pad = rows_t >= dr["counts"].view(E, 1)
        assert torch.all(got.view(torch.int16)[pad] == SENTINEL), f"replay {r}: padding written"
        if r % 5 == 0:
            c = dr["counts"].cpu().numpy()
            rows = []
            for e in range(E):
                if c[e] > 0:
                    pick = {0, int(c[e]) - 1} | set(int(v) for v in rng.choice(c[e], min(2, c[e]),
                                                                          replace=False))
                    rows += [(e, rr) for rr in sorted(pick)]
            rows = np.array(rows, np.int32)
            W = oracle_weights(cfg, w1, w2, np.unique(rows[:, 0]))
            _check_rows(cfg, {"x_b": dr["x_b"], "counts": dr["counts"]}, got, W, rows=rows)
            checked += 1
    assert checked == 4
