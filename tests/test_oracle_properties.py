"""Property checks of the oracle's sampler and quantizer over random inputs (hypothesis)."""
import numpy as np
import pytest

import oracle

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings


@settings(max_examples=60, deadline=None)
@given(n=st.integers(1, 64), k=st.integers(1, 80), temp=st.floats(0.05, 3.0), u=st.floats(0.0, 0.999999),
       seed=st.integers(0, 2 ** 31 - 1), ties=st.booleans())
def test_sampler_draws_a_candidate(n, k, temp, u, seed, ties):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal(n)
    if ties:
        lg = np.round(lg, 1)  # many equal logits
    tok = oracle.sample_topk(lg, temp, k, u)
    cand = sorted(range(n), key=lambda i: (-lg[i], i))[:min(k, n)]
    assert tok in cand
    if k == 1:
        assert tok == cand[0]


@settings(max_examples=30, deadline=None)
@given(T=st.integers(1, 6), D=st.integers(1, 12), Cb=st.integers(1, 20), seed=st.integers(0, 2 ** 31 - 1))
def test_rvq_stage0_is_a_nearest_codeword(T, D, Cb, seed):
    rng = np.random.default_rng(seed)
    zs = rng.standard_normal((T, D)).astype(np.float32)
    za = rng.standard_normal((T, D)).astype(np.float32)
    cb = rng.standard_normal((8, Cb, D)).astype(np.float32)
    codes, gap = oracle.rvq_encode(zs, za, cb)
    assert ((codes >= 0) & (codes < Cb)).all() and (gap >= 0).all()
    d = ((zs[:, None, :].astype(np.float64) - cb[0][None].astype(np.float64)) ** 2).sum(-1)
    best = d[np.arange(T), codes[:, 0]]
    assert (best <= d.min(axis=1) + 1e-9).all()
