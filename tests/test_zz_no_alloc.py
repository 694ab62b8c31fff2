"""moe_align_permute_no_ws: the counting sort for callers that cannot give
the library scratch memory (a plugin interface that passes only inputs and
outputs, or an engine whose device memory is all reserved up front).  It
must agree bit for bit with moe_align_permute, which takes a workspace, on
two calls in a row (the second call reuses the library's fixed array that
the first one left filled), and must refuse sizes beyond its fixed limit.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def g():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_count_gb300 as lib
    import oracle
    lib.load()
    oracle.build()
    return lib


def _ids(M, k, E, seed):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    return torch.from_numpy(rng.choice(E, size=(M, k), p=p / p.sum()).astype(np.int32)).to(DEV)


def _outputs(M, k, E):
    return (torch.full((E,), -1, dtype=torch.int32, device=DEV),
            torch.full((E + 1,), -1, dtype=torch.int32, device=DEV),
            torch.full((M * k,), -1, dtype=torch.int32, device=DEV),
            torch.full((M * k,), -9, dtype=torch.int32, device=DEV))


def test_no_ws_matches_workspace_version_on_two_calls_in_a_row(g):
    cases = [(8192, 8, 256, 1), (300, 2, 8, 2)]  # the second call is smaller
    for M, k, E, seed in cases:
        ids = _ids(M, k, E, seed)
        ref = _outputs(M, k, E)
        ws = g.workspace(g.WS_ALIGN, M, E, 0, 0, k, 0)
        g.moe_align_permute(ids, E, *ref, ws)
        got = _outputs(M, k, E)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        g.moe_align_permute_no_ws(ids, E, *got, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        for a, b, name in zip(ref, got, ("counts", "offsets", "sorted", "inv")):
            assert torch.equal(a, b), f"{name} differs (M={M}, E={E})"
        # and against the oracle's stable counting sort
        import oracle
        rc, bad = oracle.count(ids.cpu().numpy(), E)
        ro, rs, ri = oracle.align(ids.cpu().numpy(), E)
        assert bad == 0
        assert np.array_equal(got[0].cpu().numpy(), rc)
        assert np.array_equal(got[1].cpu().numpy(), ro)
        assert np.array_equal(got[2].cpu().numpy(), rs)
        assert np.array_equal(got[3].cpu().numpy(), ri)


def test_no_ws_refuses_sizes_beyond_its_fixed_array(g):
    M, k, E = 65536, 8, 512  # 256 chunks x 512 experts > 65536 entries
    ids = torch.zeros((M, k), dtype=torch.int32, device=DEV)
    out = _outputs(M, k, E)
    with pytest.raises(g.GbmoeError) as ei:
        g.moe_align_permute_no_ws(ids, E, *out)
    assert ei.value.status == 1  # GBMOE_INVALID_ARG, nothing enqueued
    torch.cuda.synchronize()
    assert torch.all(out[2] == -1)
