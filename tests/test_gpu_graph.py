"""The Standard-format layer captured in a CUDA graph: no call of the path
reads anything on the host, so the one-call forward can be captured once and
replayed with fresh inputs copied into its static buffers; every replay must
equal the eager call bit for bit (the capture-and-replay pattern of the
worst-tokens test, applied to the Standard format)."""
import pytest
import torch

import workloads as WL
from gpu_common import GpuWeights, gbmoe

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


@pytest.mark.parametrize("cfg", [WL.SMALL_SIGMOID, WL.SMALL_FP8, WL.SMALL_PAIR_TOP2,
                                 WL.SMALL_FP8CH, WL.SMALL_FP8T], ids=lambda c: c.name)
def test_forward_graph_replay_equals_eager(cfg):
    g = gbmoe()
    d0 = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d0["w1"], d0["w2"])
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    x = d0["x"].clone()
    logits = d0["logits"].clone()
    bias = d0["bias"]
    out = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype)

    def fwd(xx, ll, oo):
        g.moe_forward(xx, ll, bias, N, E, k, cfg.score_fn, cfg.n_groups, cfg.topk_groups,
                      cfg.renorm, cfg.dtype, gw.w1, gw.w1s, gw.w2, gw.w2s, oo, ws,
                      err_word=err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fwd(x, logits, out)  # first call outside the capture (one-time set-up)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd(x, logits, out)
    for r in range(3):
        dr = WL.make_inputs(cfg, DEV, seed=cfg.seed + 100 + r, with_weights=False)
        x.copy_(dr["x"])
        logits.copy_(dr["logits"])
        graph.replay()
        eager = torch.empty_like(out)
        fwd(dr["x"], dr["logits"], eager)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16)), f"replay {r}"
