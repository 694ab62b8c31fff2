"""Checks the GPU tests rely on, pinned on the CPU.  The near-tie validity
check: the oracle's own choice passes, a wrong expert or a wrong group fails,
and when two group keys tie within the tolerance both group choices pass (and
only those).  The guard-band allocator: writes inside its buffers pass, one
byte written just before or just past a buffer fails."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_common import GUARD, Guarded, _grouped_choice_is_valid


def _route_one(v, topk, n_groups, topk_groups):
    ids, _, margin = orc.route(v[None, :].astype(np.float32), None, topk, orc.SIGMOID,
                               n_groups, topk_groups, True)
    return ids[0], margin[0]


def test_oracle_choice_is_valid_and_perturbations_are_not(orc):
    rng = np.random.default_rng(5)
    for _ in range(40):
        v = rng.standard_normal(64).astype(np.float32)
        ids, _ = _route_one(v, 6, 8, 4)
        assert _grouped_choice_is_valid(v, ids, 6, 8, 4, 1e-6)
        # the last pick swapped for the best expert left out of its group set
        gs = 8
        groups = set(int(e) // gs for e in ids)
        rest = [e for e in range(64) if e // gs in groups and e not in ids]
        worse = ids.copy()
        worse[-1] = rest[0]
        assert not _grouped_choice_is_valid(v, worse, 6, 8, 4, 1e-6)
        # an expert from a group that was not kept
        out_group = [e for e in range(64) if e // gs not in groups]
        bad = ids.copy()
        bad[-1] = out_group[0]
        assert not _grouped_choice_is_valid(v, bad, 6, 8, 4, 1e-6)
        # order matters: ids come in descending value order
        assert not _grouped_choice_is_valid(v, ids[::-1].copy(), 6, 8, 4, 1e-6)


def test_tied_group_keys_accept_either_group(orc):
    # 4 groups of 4, keep 1 group, top-2: groups 1 and 3 hold the same two
    # largest values (equal keys), so either group is a correct result; the
    # oracle takes the lower group index
    v = np.array([-3, -3, -3, -3, 2.0, 1.0, -5, -5, -3, -3, -3, -3, -4, 1.0, 2.0, -4],
                 np.float32)
    ids, margin = _route_one(v, 2, 4, 1)
    assert list(ids) == [4, 5] and margin == 0.0
    assert _grouped_choice_is_valid(v, np.array([4, 5]), 2, 4, 1, 1e-6)
    assert _grouped_choice_is_valid(v, np.array([14, 13]), 2, 4, 1, 1e-6)
    assert not _grouped_choice_is_valid(v, np.array([13, 14]), 2, 4, 1, 1e-6)
    assert not _grouped_choice_is_valid(v, np.array([4, 14]), 2, 4, 1, 1e-6)
    # with the tie broken by more than the tolerance only group 1 is valid
    v2 = v.copy()
    v2[13] = 0.9
    assert not _grouped_choice_is_valid(v2, np.array([14, 13]), 2, 4, 1, 1e-6)


def test_guard_bands_catch_a_write_just_outside_a_buffer():
    guard = Guarded(device="cpu")
    a = guard((3, 5), torch.float32)
    b = guard((7,), torch.bfloat16)
    a.fill_(1.0)
    b.fill_(2.0)
    guard.check("in bounds")
    for buf, off in ((0, -1), (0, 60), (1, 14)):  # before a, just past a, just past b
        raw = guard.bufs[buf][0]
        old = int(raw[GUARD + off])
        raw[GUARD + off] = 0
        with pytest.raises(AssertionError):
            guard.check("planted")
        raw[GUARD + off] = old
    guard.check("restored")
