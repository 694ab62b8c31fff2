"""moe_grouped_gemm_down_reduce: the down GEMM with the ordered top-k reduce
in its epilogue must equal moe_grouped_gemm_down followed by
moe_unpermute_weighted_reduce bit for bit (slot rows and output), on every
kernel the down GEMM dispatches to, on an expert-parallel shard whose tokens
partly have no local slot (their rows must come out zero), and on repeated
calls that reuse one workspace (the counters are cleared by each call)."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import GpuWeights, gbmoe

pytestmark = pytest.mark.gpu

DEV = "cuda"
GARBAGE = 0x7FC1  # a bf16 NaN: any row the call fails to write stays NaN


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


def _hidden(cfg, g, d, ids, offsets, srt, gw):
    """Gate/up on the GPU: H (and its scales) in the layout the down GEMM takes."""
    M, E, N, K, k, P = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk, cfg.P
    ld = (P + 3) // 4 * 4
    if cfg.dtype == WL.BF16:
        A = torch.empty((P, K), dtype=torch.bfloat16, device=DEV)
        g.moe_permute_rows(d["x"], None, srt, offsets, k, E, cfg.dtype, A, None)
        H = torch.empty((P, N), dtype=torch.bfloat16, device=DEV)
        g.moe_grouped_gemm_gate_up_silu(A, None, offsets, M, k, E, N, K, gw.w1, None,
                                        cfg.dtype, H, None)
        return H, None
    ch = cfg.dtype == WL.FP8_CHANNEL
    sk = 1 if ch else K // 128
    xq = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    xs = torch.empty((M, sk), dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_group(d["x"], xq, xs, group=K if ch else 128)
    A = torch.empty((P, K), dtype=torch.uint8, device=DEV)
    As = torch.empty((sk, ld), dtype=torch.float32, device=DEV)
    g.moe_permute_rows(xq, xs, srt, offsets, k, E, cfg.dtype, A, As)
    if ch:
        Hb = torch.empty((P, N), dtype=torch.bfloat16, device=DEV)
        g.moe_grouped_gemm_gate_up_silu(A, As, offsets, M, k, E, N, K, gw.w1, gw.w1s,
                                        cfg.dtype, Hb, None)
        H = torch.empty((P, N), dtype=torch.uint8, device=DEV)
        Hs = torch.empty((P, 1), dtype=torch.float32, device=DEV)
        g.moe_quant_fp8_group(Hb, H, Hs, group=N)
        return H, Hs
    H = torch.empty((P, N), dtype=torch.uint8, device=DEV)
    Hs = torch.empty((N // 128, ld), dtype=torch.float32, device=DEV)
    g.moe_grouped_gemm_gate_up_silu(A, As, offsets, M, k, E, N, K, gw.w1, gw.w1s, cfg.dtype,
                                    H, Hs)
    return H, Hs


def _compare(cfg, d, gw, ids, wts, expert_map=None, E_global=None, repeats=2):
    g = gbmoe()
    M, E, N, K, k, P = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk, cfg.P
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    srt = torch.empty(P, dtype=torch.int32, device=DEV)
    inv = torch.empty(P, dtype=torch.int32, device=DEV)
    g.moe_align_permute(ids, E, None, offsets, srt, inv,
                        g.workspace(g.WS_ALIGN, M, E, 0, 0, k, 0), expert_map=expert_map,
                        E_global=E_global)
    H, Hs = _hidden(cfg, g, d, ids, offsets, srt, gw)
    y_ref = torch.zeros((M, k, K), dtype=torch.bfloat16, device=DEV)
    out_ref = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    g.moe_grouped_gemm_down(H, Hs, srt, offsets, wts, M, k, E, N, K, gw.w2, gw.w2s, cfg.dtype,
                            y_ref)
    g.moe_unpermute_weighted_reduce(y_ref, inv, M, k, K, out_ref)
    ws = g.workspace(g.WS_DOWN_REDUCE, M, E, N, K, k, cfg.dtype)
    for r in range(repeats):
        y = torch.zeros((M, k, K), dtype=torch.bfloat16, device=DEV)
        out = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
        out.view(torch.int16).fill_(GARBAGE)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        g.moe_grouped_gemm_down_reduce(H, Hs, srt, inv, offsets, wts, M, k, E, N, K, gw.w2,
                                       gw.w2s, cfg.dtype, y, out, ws, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), f"{cfg.name} y, call {r}"
        assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16)), \
            f"{cfg.name} out, call {r}"
    return inv, out_ref


CASES = [WL.TINY, WL.SMALL_BF16, WL.SMALL_SIGMOID, WL.SMALL_FP8, WL.SMALL_PAIR,
         WL.SMALL_PAIR_TOP2, WL.SMALL_FP8_K640, WL.SMALL_FP8CH, WL.SMALL_FP8CH_PAIR]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_down_reduce_equals_down_then_reduce(cfg):
    d = WL.make_inputs(cfg, DEV)
    rid, rw, _ = orc.route(d["logits"].cpu().numpy(),
                           None if d["bias"] is None else d["bias"].cpu().numpy(),
                           cfg.topk, cfg.score_fn, cfg.n_groups, cfg.topk_groups, cfg.renorm)
    ids = torch.from_numpy(rid).to(DEV)
    wts = torch.from_numpy(rw.astype(np.float32)).to(DEV)
    _compare(cfg, d, GpuWeights(cfg, d["w1"], d["w2"]), ids, wts)


@pytest.mark.parametrize("dtype", [WL.BF16, WL.FP8_CHANNEL], ids=["bf16", "fp8ch"])
def test_down_reduce_on_a_shard_zeroes_tokens_without_local_slots(dtype):
    """12 of 64 routed experts on this shard, top-4: about a third of the
    tokens have no local slot; their output rows are zero."""
    base = WL.MoEConfig("ep_fused", M=300, K=384, N=256, E=64, topk=4, dtype=dtype, seed=61)
    d = WL.make_inputs(base, DEV)
    rng = np.random.default_rng(61)
    local = np.sort(rng.choice(64, 12, replace=False))
    emap = np.full(64, -1, np.int32)
    emap[local] = np.arange(12, dtype=np.int32)
    rid, rw, _ = orc.route(d["logits"].cpu().numpy(), None, 4, orc.SOFTMAX, 1, 1, True)
    lcfg = WL.MoEConfig("ep_fused_local", M=300, K=384, N=256, E=12, topk=4, dtype=dtype,
                        seed=61)
    sel = torch.from_numpy(local).to(DEV)
    gw = GpuWeights(lcfg, d["w1"][sel].contiguous(), d["w2"][sel].contiguous())
    inv, out = _compare(lcfg, d, gw, torch.from_numpy(rid).to(DEV),
                        torch.from_numpy(rw.astype(np.float32)).to(DEV),
                        expert_map=torch.from_numpy(emap).to(DEV), E_global=64)
    none_local = ~np.isin(rid, local).any(1)
    assert none_local.sum() > 20
    assert torch.all(out[torch.from_numpy(np.flatnonzero(none_local)).to(DEV)].float() == 0)
    assert np.array_equal(inv.cpu().numpy().reshape(300, 4) >= 0, np.isin(rid, local))
