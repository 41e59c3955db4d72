"""Property tests of the oracle's routing and dispatch over random shapes (CPU only).

Hypothesis draws the shape (T, E, k) and logits from a small value set, so that ties, +0 and
-0 occur often; each draw is checked against numpy's lexsort (descending logit, then
ascending index, +0 == -0), the closed-form softmax of the selected logits, and the dispatch
invariants: counts sum to T k, offsets are their exclusive prefix sum, perm is a bijection
ordered by (expert, token) and pos is its inverse.  Skipped where hypothesis is not
installed.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402

_VALUES = [-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 3.0]


@st.composite
def _problems(draw):
    E = draw(st.integers(1, 24))
    k = draw(st.integers(1, min(E, 16)))
    T = draw(st.integers(0, 12))
    vals = draw(st.lists(st.sampled_from(_VALUES), min_size=T * E, max_size=T * E))
    return np.array(vals, np.float32).reshape(T, E), k


@settings(max_examples=150, deadline=None)
@given(_problems())
def test_route_and_dispatch_properties(problem):
    logits, k = problem
    T, E = logits.shape
    idx, gate = oracle.route(logits, k)
    assert idx.shape == (T, k) and gate.shape == (T, k)
    for t in range(T):
        # -x turns -0.0 into +0.0 and +0.0 into -0.0; both compare equal in the sort keys
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        assert idx[t].tolist() == order[:k].tolist()
        sel = logits[t, order[:k]].astype(np.float64)
        ref = np.exp(sel - sel.max())
        np.testing.assert_allclose(gate[t], ref / ref.sum(), rtol=1e-14, atol=1e-300)
    counts, offsets, perm, pos = oracle.dispatch(idx, E)
    P = T * k
    assert counts.tolist() == np.bincount(idx.reshape(-1), minlength=E).tolist()
    assert offsets.tolist() == [0] + np.cumsum(counts).tolist()
    assert sorted(perm.tolist()) == list(range(P))
    assert (pos[perm] == np.arange(P)).all()
    keys = [(int(idx.reshape(-1)[p]), int(p) // k) for p in perm]
    assert keys == sorted(keys)                      # rows ordered by (expert, token)
