"""expert_map and apply_router_weight_on_input (the expert-parallel and
weight-placement options of FusedMoEModularKernel.forward) against the
oracle: counts and permutation bit-exact, layer outputs within tolerance."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as WL
from gpu_common import TOL, GpuWeights, assert_close_rel, gbmoe

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


def _shard_map(Eg, local, seed=0):
    emap = np.full(Eg, -1, np.int32)
    emap[np.asarray(local)] = np.arange(len(local), dtype=np.int32)
    return emap


def test_count_align_with_expert_map_bit_exact():
    g = gbmoe()
    rng = np.random.default_rng(40)
    Eg, M, k = 64, 777, 6
    local = np.sort(rng.choice(Eg, 23, replace=False))
    emap = _shard_map(Eg, local)
    El = len(local)
    ids_np = rng.integers(0, Eg, (M, k)).astype(np.int32)
    ids_np[5, 0] = Eg + 3  # invalid
    ids = torch.from_numpy(ids_np).to(DEV)
    m = torch.from_numpy(emap).to(DEV)
    counts = torch.full((El,), -7, dtype=torch.int32, device=DEV)
    counts2 = torch.full((El,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.empty(El + 1, dtype=torch.int32, device=DEV)
    srt = torch.full((M * k,), -5, dtype=torch.int32, device=DEV)
    inv = torch.empty(M * k, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_ALIGN, M, El, 0, 0, k, 0)
    g.moe_count_expert_tokens(ids, El, counts, err, expert_map=m, E_global=Eg)
    g.moe_align_permute(ids, El, counts2, offsets, srt, inv, ws, err, expert_map=m, E_global=Eg)
    torch.cuda.synchronize()
    rc, bad = orc.count(ids_np, Eg, emap, El)
    ro, rs, ri = orc.align(ids_np, Eg, emap, El)
    assert bad == 1 and err.item() & g.ERR_BAD_EXPERT_ID
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(counts2.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(srt.cpu().numpy()[: ro[El]], rs)
    assert np.array_equal(inv.cpu().numpy(), ri)


@pytest.mark.parametrize("dtype", [WL.BF16, WL.FP8, WL.FP8_CHANNEL, WL.FP8_TENSOR],
                         ids=["bf16", "fp8", "fp8ch", "fp8t"])
def test_forward_on_an_expert_parallel_shard(dtype):
    """The shard holding 24 of 64 routed experts: its output is the local
    part of the layer (non-local slots add nothing)."""
    g = gbmoe()
    base = WL.MoEConfig("ep", M=200, K=384, N=256, E=64, topk=6, dtype=dtype,
                        score_fn=WL.SIGMOID, n_groups=8, topk_groups=4,
                        zipf_bias=True, seed=41)
    d = WL.make_inputs(base, DEV)
    rng = np.random.default_rng(41)
    local = np.sort(rng.choice(64, 24, replace=False))
    emap = _shard_map(64, local)
    lcfg = WL.MoEConfig("ep_local", M=200, K=384, N=256, E=24, topk=6, dtype=dtype, seed=41)
    lw1 = d["w1"][torch.from_numpy(local).to(DEV)].contiguous()
    lw2 = d["w2"][torch.from_numpy(local).to(DEV)].contiguous()
    gw = GpuWeights(lcfg, lw1, lw2)
    out = torch.empty((base.M, base.K), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_FORWARD, base.M, 24, base.N, base.K, base.topk, dtype)
    g.moe_forward(d["x"], d["logits"], d["bias"], base.N, 24, base.topk, base.score_fn,
                  base.n_groups, base.topk_groups, True, dtype, gw.w1, gw.w1s, gw.w2, gw.w2s,
                  out, ws, err_word=err, expert_map=torch.from_numpy(emap).to(DEV))
    torch.cuda.synchronize()
    assert err.item() == 0
    from gpu_common import oracle_weights
    W = oracle_weights(lcfg, lw1, lw2)
    ref, _, _ = orc.moe_forward(WL.bf16_bits(d["x"]), d["logits"].cpu().numpy(),
                                d["bias"].cpu().numpy(), base.topk, orc.SIGMOID, W,
                                base.n_groups, base.topk_groups, True, base.requant_h,
                                expert_map=emap)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[dtype], "shard")


@pytest.mark.parametrize("dtype", [WL.BF16, WL.FP8, WL.FP8_CHANNEL, WL.FP8_TENSOR],
                         ids=["bf16", "fp8", "fp8ch", "fp8t"])
def test_forward_with_router_weight_on_input(dtype):
    """Top-1, unrenormalised softmax weights p < 1: out = expert(p x)."""
    g = gbmoe()
    cfg = WL.MoEConfig("woi", M=150, K=256, N=256, E=8, topk=1, dtype=dtype, renorm=False,
                       seed=42)
    d = WL.make_inputs(cfg, DEV)
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    out = torch.empty((cfg.M, cfg.K), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((cfg.M, 1), dtype=torch.int32, device=DEV)
    wts = torch.empty((cfg.M, 1), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = g.workspace(g.WS_FORWARD, cfg.M, cfg.E, cfg.N, cfg.K, 1, dtype)
    g.moe_forward(d["x"], d["logits"], None, cfg.N, cfg.E, 1, cfg.score_fn, 1, 1, False, dtype,
                  gw.w1, gw.w1s, gw.w2, gw.w2s, out, ws, topk_ids=ids, topk_weights=wts,
                  err_word=err, apply_router_weight_on_input=True)
    torch.cuda.synchronize()
    assert err.item() == 0
    from gpu_common import oracle_weights
    W = oracle_weights(cfg, d["w1"], d["w2"])
    ref, rid, rw = orc.moe_forward(WL.bf16_bits(d["x"]), d["logits"].cpu().numpy(), None, 1,
                                   orc.SOFTMAX, W, renorm=False, requant_h=cfg.requant_h,
                                   weight_on_input=True)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[dtype], "weight on input")


def test_quant_with_row_weights_bit_exact():
    g = gbmoe()
    gen = torch.Generator(device=DEV).manual_seed(43)
    x = torch.randn((99, 512), generator=gen, device=DEV).to(torch.bfloat16)
    rw = torch.rand(99, generator=gen, device=DEV)
    q = torch.empty((99, 512), dtype=torch.uint8, device=DEV)
    s = torch.empty((99, 4), dtype=torch.float32, device=DEV)
    g.moe_quant_fp8_group(x, q, s, row_weights=rw)
    rq, rs = orc.quant_fp8_group(WL.bf16_bits(x), row_weights=rw.cpu().numpy())
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)
