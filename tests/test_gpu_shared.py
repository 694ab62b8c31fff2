"""Shared experts (a dense gated MLP on every token, returned beside the
routed output), in bf16 or in e4m3 with block-scaled weights, and their
overlap with the routed experts on an auxiliary stream, the
MULTI_STREAM_OVERLAPPED order of the SharedExperts page."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import TOL, GpuWeights, assert_close_rel, gbmoe

pytestmark = pytest.mark.gpu

DEV = "cuda"
NS = 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


def _shared_weights(K, Ns, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    w1s = (torch.randn((2 * Ns, K), generator=g, device=DEV) / K ** 0.5).to(torch.bfloat16)
    w2s = (torch.randn((K, Ns), generator=g, device=DEV) / Ns ** 0.5).to(torch.bfloat16)
    return w1s, w2s


@pytest.mark.parametrize("act", [0, 1], ids=["silu", "gelu"])
def test_shared_expert_is_the_dense_mlp(act):
    g = gbmoe()
    cfg = WL.SMALL_BF16
    d = WL.make_inputs(cfg, DEV, with_weights=False)
    w1s, w2s = _shared_weights(cfg.K, NS, 50)
    out_s = torch.empty((cfg.M, cfg.K), dtype=torch.bfloat16, device=DEV)
    ws = g.workspace(g.WS_SHARED, cfg.M, 1, NS, cfg.K, 1, g.BF16)
    g.moe_shared_expert_forward(d["x"], NS, w1s, w2s, out_s, ws, activation=act)
    torch.cuda.synchronize()
    # the oracle's batched form with one expert holding every token
    W = orc.Weights(orc.BF16, WL.bf16_bits(w1s)[None], WL.bf16_bits(w2s)[None], act=act)
    ref, n = orc.batched_experts(WL.bf16_bits(d["x"])[None], np.array([cfg.M], np.int32), W)
    assert n == cfg.M
    assert_close_rel(out_s.float().cpu().numpy(), ref[0], TOL[WL.BF16], "shared")


def _shared_e4m3(w1s, w2s):
    """The library's 128 x 128 block quantisation of the shared weights:
    (w1 codes, w1 scales, w2 codes, w2 scales)."""
    g = gbmoe()
    (Ns2, K), Ns = w1s.shape, w2s.shape[1]
    q1 = torch.empty((Ns2, K), dtype=torch.uint8, device=DEV)
    s1 = torch.empty((Ns2 // 128, K // 128), dtype=torch.float32, device=DEV)
    q2 = torch.empty((K, Ns), dtype=torch.uint8, device=DEV)
    s2 = torch.empty((K // 128, Ns // 128), dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_block(w1s, q1, s1)
    g.moe_quant_fp8_block(w2s, q2, s2)
    return q1, s1, q2, s2


def _shared_e4m3_channel(w1s, w2s):
    """The library's per-row (per output channel) quantisation of the shared
    weights: (w1 codes, w1 scales (2Ns), w2 codes, w2 scales (K))."""
    g = gbmoe()
    (Ns2, K), Ns = w1s.shape, w2s.shape[1]
    q1 = torch.empty((Ns2, K), dtype=torch.uint8, device=DEV)
    s1 = torch.empty((Ns2, 1), dtype=torch.float32, device=DEV)
    q2 = torch.empty((K, Ns), dtype=torch.uint8, device=DEV)
    s2 = torch.empty((K, 1), dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_group(w1s, q1, s1, group=K)
    g.moe_quant_fp8_group(w2s, q2, s2, group=Ns)
    return q1, s1.view(-1), q2, s2.view(-1)


@pytest.mark.parametrize("cfg,act,dtype",
                         [(WL.SMALL_BF16, 0, WL.FP8), (WL.SMALL_BF16, 1, WL.FP8),
                          (WL.SMALL_FP8_K640, 0, WL.FP8), (WL.SMALL_BF16, 0, WL.FP8_CHANNEL),
                          (WL.SMALL_FP8_K640, 1, WL.FP8_CHANNEL)],
                         ids=["block_M300_K512_silu", "block_M300_K512_gelu", "block_M300_K640_silu",
                              "channel_M300_K512_silu", "channel_M300_K640_gelu"])
def test_shared_expert_e4m3_is_the_oracles_e4m3_mlp(cfg, act, dtype):
    """e4m3 shared experts against the oracle's e4m3 experts with one expert
    holding every token (ragged last m-tile; K = 640 leaves the second half
    of the last down tile past K).  Block scales: x quantised in 1 x 128
    groups inside the call, 128 x 128 weight blocks, h requantised in 1 x 128
    groups.  Per-channel: one scale per token of x and per weight row, h kept
    in bf16 and quantised per row."""
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV, with_weights=False)
    M, K = cfg.M, cfg.K
    w1s, w2s = _shared_weights(K, NS, 52)
    block = dtype == WL.FP8
    q1, s1, q2, s2 = _shared_e4m3(w1s, w2s) if block else _shared_e4m3_channel(w1s, w2s)
    out_s = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = g.workspace(g.WS_SHARED, M, 1, NS, K, 1, dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    g.moe_shared_expert_forward(d["x"], NS, q1, q2, out_s, ws, dtype=dtype, activation=act,
                                err_word=err, w1s_scales=s1, w2s_scales=s2)
    torch.cuda.synchronize()
    assert err.item() == 0
    if block:
        oq1, os1 = orc.quant_fp8_block(WL.bf16_bits(w1s))
        oq2, os2 = orc.quant_fp8_block(WL.bf16_bits(w2s))
    else:
        oq1, os1 = orc.quant_fp8_group(WL.bf16_bits(w1s), group=K)
        oq2, os2 = orc.quant_fp8_group(WL.bf16_bits(w2s), group=NS)
        os1, os2 = os1[:, 0], os2[:, 0]
    # the weights the GPU ran with are the oracle's own quantisation
    assert np.array_equal(q1.cpu().numpy(), oq1) and np.array_equal(q2.cpu().numpy(), oq2)
    assert np.array_equal(s1.cpu().numpy(), os1) and np.array_equal(s2.cpu().numpy(), os2)
    W = orc.Weights(dtype, experts={0: (oq1, oq2, os1, os2)}, E=1, N=NS, K=K, act=act)
    ref, n = orc.batched_experts(WL.bf16_bits(d["x"])[None], np.array([M], np.int32), W,
                                 requant_h=True)
    assert n == M
    assert_close_rel(out_s.float().cpu().numpy(), ref[0], TOL[dtype], f"shared e4m3 ({dtype})")


@pytest.mark.parametrize("cfg,shared_dtype,ns",
                         [(WL.SMALL_SIGMOID, WL.BF16, NS), (WL.SMALL_FP8, WL.FP8, NS),
                          (WL.SMALL_FP8CH, WL.FP8_CHANNEL, NS),
                          # the DeepSeek-V3-shaped e4m3 layer and shared expert the bench times
                          (WL.DSV3_PREFILL_FP8, WL.FP8, 2048)],
                         ids=["bf16", "e4m3", "e4m3_channel", "e4m3_full_size"])
def test_overlapped_shared_experts_equal_the_separate_calls_and_replay(cfg, shared_dtype, ns):
    """moe_forward_shared (routed experts on the caller's stream, the shared
    expert on an auxiliary stream between two caller events) equals the two
    separate calls on one stream bit for bit, eagerly and as a CUDA graph
    replayed with new tokens."""
    NS = ns
    g = gbmoe()
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    w1s, w2s = _shared_weights(cfg.K, NS, 51)
    s1 = s2 = None
    if shared_dtype == WL.FP8:
        w1s, s1, w2s, s2 = _shared_e4m3(w1s, w2s)
    elif shared_dtype == WL.FP8_CHANNEL:
        w1s, s1, w2s, s2 = _shared_e4m3_channel(w1s, w2s)
    sh = dict(dtype=shared_dtype, w1s_scales=s1, w2s_scales=s2)
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    ws = g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype)
    ws_s = g.workspace(g.WS_SHARED, M, 1, NS, K, 1, shared_dtype)
    args = (d["logits"], d["bias"], N, E, k, cfg.score_fn, cfg.n_groups, cfg.topk_groups,
            cfg.renorm, cfg.dtype, gw.w1, gw.w1s, gw.w2, gw.w2s)
    # separate calls on one stream
    ref_out = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    ref_sh = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    g.moe_forward(d["x"], *args, ref_out, ws)
    g.moe_shared_expert_forward(d["x"], NS, w1s, w2s, ref_sh, ws_s, **sh)
    # overlapped
    aux = torch.cuda.Stream()
    ev_in = torch.cuda.Event()
    ev_out = torch.cuda.Event()
    x = d["x"].clone()
    out = torch.empty_like(ref_out)
    out_sh = torch.empty_like(ref_sh)
    ws2 = g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype)
    ws2_s = g.workspace(g.WS_SHARED, M, 1, NS, K, 1, shared_dtype)

    def run():
        g.moe_forward_shared(x, *args, out, ws2, NS, w1s, w2s, out_sh, ws2_s,
                             aux_stream=aux, ev_input_ready=ev_in, ev_output_ready=ev_out,
                             shared_dtype=shared_dtype, w1s_scales=s1, w2s_scales=s2)

    run()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(out_sh.view(torch.int16), ref_sh.view(torch.int16))
    # the fork/join captured in a CUDA graph, replayed with new tokens
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    x2 = WL.make_inputs(cfg, DEV, seed=cfg.seed + 7, with_weights=False)["x"]
    x.copy_(x2)
    graph.replay()
    torch.cuda.synchronize()
    g.moe_forward(x2, *args, ref_out, ws)
    g.moe_shared_expert_forward(x2, NS, w1s, w2s, ref_sh, ws_s, **sh)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(out_sh.view(torch.int16), ref_sh.view(torch.int16))


def test_shared_expert_e4m3_full_size_sampled():
    """The DeepSeek-V3-shaped shared expert (K = 7168, Ns = 2048) on 8192
    tokens in e4m3: 512 seeded rows plus the first and the last against the
    oracle's e4m3 expert, and the whole output finite."""
    g = gbmoe()
    M, K, Ns = 8192, 7168, 2048
    gen = torch.Generator(device=DEV).manual_seed(53)
    x = torch.randn((M, K), generator=gen, device=DEV).to(torch.bfloat16)
    w1s, w2s = _shared_weights(K, Ns, 54)
    q1, s1, q2, s2 = _shared_e4m3(w1s, w2s)
    out_s = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    ws = g.workspace(g.WS_SHARED, M, 1, Ns, K, 1, g.FP8_E4M3)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    g.moe_shared_expert_forward(x, Ns, q1, q2, out_s, ws, dtype=g.FP8_E4M3, err_word=err,
                                w1s_scales=s1, w2s_scales=s2)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert bool(torch.isfinite(out_s.float()).all())
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(55).choice(M, 512, replace=False)]))
    oq1, os1 = orc.quant_fp8_block(WL.bf16_bits(w1s))
    oq2, os2 = orc.quant_fp8_block(WL.bf16_bits(w2s))
    W = orc.Weights(WL.FP8, experts={0: (oq1, oq2, os1, os2)}, E=1, N=Ns, K=K)
    sel = np.stack([np.zeros_like(rows), rows], 1)
    ref, n = orc.batched_experts(WL.bf16_bits(x)[None], np.array([M], np.int32), W,
                                 rows=sel, requant_h=True)
    assert n == len(rows)
    got = out_s.float().cpu().numpy()
    assert_close_rel(got[rows], ref[0][rows], TOL[WL.FP8], "shared e4m3 full size")
