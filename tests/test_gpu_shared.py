"""Shared experts (a dense gated MLP on every token, returned beside the
routed output) and their overlap with the routed experts on an auxiliary
stream, the MULTI_STREAM_OVERLAPPED order of the SharedExperts page."""
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


def test_overlapped_shared_experts_equal_the_separate_calls_and_replay():
    g = gbmoe()
    cfg = WL.SMALL_SIGMOID
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    w1s, w2s = _shared_weights(cfg.K, NS, 51)
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    ws = g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype)
    ws_s = g.workspace(g.WS_SHARED, M, 1, NS, K, 1, g.BF16)
    args = (d["logits"], d["bias"], N, E, k, cfg.score_fn, cfg.n_groups, cfg.topk_groups,
            cfg.renorm, cfg.dtype, gw.w1, gw.w1s, gw.w2, gw.w2s)
    # separate calls on one stream
    ref_out = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    ref_sh = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    g.moe_forward(d["x"], *args, ref_out, ws)
    g.moe_shared_expert_forward(d["x"], NS, w1s, w2s, ref_sh, ws_s)
    # overlapped
    aux = torch.cuda.Stream()
    ev_in = torch.cuda.Event()
    ev_out = torch.cuda.Event()
    x = d["x"].clone()
    out = torch.empty_like(ref_out)
    out_sh = torch.empty_like(ref_sh)
    ws2 = g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype)
    ws2_s = g.workspace(g.WS_SHARED, M, 1, NS, K, 1, g.BF16)

    def run():
        g.moe_forward_shared(x, *args, out, ws2, NS, w1s, w2s, out_sh, ws2_s,
                             aux_stream=aux, ev_input_ready=ev_in, ev_output_ready=ev_out)

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
    g.moe_shared_expert_forward(x2, NS, w1s, w2s, ref_sh, ws_s)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(out_sh.view(torch.int16), ref_sh.view(torch.int16))
