"""Failure detection on the GPU without a GPU fault: the bounded pipeline wait
that every GEMM kernel uses gives up on a barrier nothing completes, reports
GBMOE_ERR_TIMEOUT through the caller's error word, and leaves the context
usable (a layer run afterwards still matches the oracle)."""
import time

import numpy as np
import pytest
import torch

import workloads as WL
from gpu_common import (TOL, GpuWeights, assert_close_rel, gbmoe, oracle_forward,
                        oracle_weights, run_forward)

pytestmark = pytest.mark.gpu

GBMOE_ERR_TIMEOUT = 0x4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gbmoe()


@pytest.mark.parametrize("limit_us", [1000, 20000])
def test_bounded_wait_gives_up_and_flags_timeout(limit_us):
    g = gbmoe()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.gbmoe_selftest_bounded_wait(err, limit_us)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert err.item() == GBMOE_ERR_TIMEOUT
    # it waited at least its limit, and gave up well before a hang
    assert waited >= limit_us * 1e-6
    assert waited < 1.0


def test_context_usable_after_a_timed_out_wait():
    g = gbmoe()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g.gbmoe_selftest_bounded_wait(err, 1000)
    torch.cuda.synchronize()
    assert err.item() == GBMOE_ERR_TIMEOUT
    cfg = WL.TINY
    d = WL.make_inputs(cfg, "cuda")
    gw = GpuWeights(cfg, d["w1"], d["w2"])
    out, ids, _, lerr = run_forward(cfg, d, gw)
    torch.cuda.synchronize()
    assert lerr.item() == 0
    ref, rid, _ = oracle_forward(cfg, d, oracle_weights(cfg, d["w1"], d["w2"]))
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert_close_rel(out.float().cpu().numpy(), ref, TOL[cfg.dtype], cfg.name)
