"""The seeded input generators (CPU): determinism and the stated properties of the
synthetic routing and draft-id lists."""
from __future__ import annotations

import numpy as np
import pytest

import workloads


def test_routing_is_deterministic_distinct_and_in_range():
    for ntok, topk, n_exp, share in [(1, 10, 512, 0.65), (4, 10, 512, 0.65), (4, 8, 16, 0.65), (3, 3, 4, 0.0),
                                     (4, 10, 512, 1.0)]:
        a = workloads.routing(7, ntok, topk, n_exp, share)
        b = workloads.routing(7, ntok, topk, n_exp, share)
        assert a.dtype == np.int32 and a.shape == (ntok, topk)
        assert np.array_equal(a, b)
        assert a.min() >= 0 and a.max() < n_exp
        for row in a:
            assert len(set(row.tolist())) == topk          # distinct experts per token


def test_routing_share_sets_the_number_of_active_experts():
    """About topk + (ntok - 1) * topk * (1 - share) experts are active in a step: share 0
    gives ntok * topk distinct experts, share 1 the first token's topk."""
    assert len(np.unique(workloads.routing(1, 4, 10, 512, 0.0))) == 40
    assert len(np.unique(workloads.routing(1, 4, 10, 512, 1.0))) == 10
    for ntok in (2, 3, 4):
        u = np.mean([len(np.unique(workloads.routing(s, ntok, 10, 512, 0.65))) for s in range(300)])
        want = 10 + (ntok - 1) * 10 * 0.35
        assert abs(u - want) < 0.4, (ntok, u, want)


def test_routing_rejects_impossible_topk():
    with pytest.raises(ValueError):
        workloads.routing(1, 2, 5, 4, 0.5)


def test_draft_ids_sorted_distinct():
    ids = workloads.draft_ids(131, 248320, 106299)
    assert ids.dtype == np.int32 and len(ids) == 106299
    assert np.all(np.diff(ids) > 0) and ids[0] >= 0 and ids[-1] < 248320


def test_expert_matrices_are_distinct_and_reproducible():
    a = workloads.expert_matrix(150, 3, 8, 64)
    assert np.array_equal(a, workloads.expert_matrix(150, 3, 8, 64))
    assert not np.array_equal(a, workloads.expert_matrix(150, 4, 8, 64))
    assert a.dtype == np.float32 and abs(float(a.std()) - 0.02) < 0.01
