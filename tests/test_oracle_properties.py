"""Property-based pins of the oracle over random small shapes (hypothesis):
the same identities as the fixed pins, drawn across sizes and chunkings so
that an index or tail mistake that a fixed shape misses still fails."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402

SETTINGS = dict(max_examples=25, deadline=None, derandomize=True)


@settings(**SETTINGS)
@given(T=st.integers(1, 37), chunk=st.sampled_from([1, 2, 3, 5, 8, 16]), H=st.integers(1, 2),
       K=st.sampled_from([2, 3, 5]), V=st.sampled_from([2, 4]), seed=st.integers(0, 2**16))
def test_chunked_form_equals_recurrence_for_any_chunking(T, chunk, H, K, V, seed):
    """Chunked KDA (model file, _torch_chunk_kda) reaches the token recurrence
    for any chunk size, including a ragged last chunk."""
    rng = np.random.default_rng(seed)
    q, k = rng.standard_normal((T, H, K)), rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = -rng.uniform(0.0, 1.0, (T, H, K))
    beta = rng.uniform(0.0, 1.0, (T, H))
    s0 = 0.3 * rng.standard_normal((H, K, V))
    o_r, s_r = oracle.recurrence(q, k, v, g, beta, initial_state=s0[None])
    o_c, s_c = oracle.chunked_form(q, k, v, g, beta, initial_state=s0, chunk=chunk)
    np.testing.assert_allclose(o_c, o_r, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(s_c, s_r[0], rtol=1e-9, atol=1e-11)


@settings(**SETTINGS)
@given(L1=st.integers(0, 12), L2=st.integers(0, 12), ks=st.integers(2, 6), D=st.integers(1, 4),
       act=st.sampled_from(["silu", "none"]), seed=st.integers(0, 2**16))
def test_short_conv_prefill_splits_through_its_final_state(L1, L2, ks, D, act, seed):
    """A prefill over L1 + L2 tokens equals a prefill over L1 followed by a
    prefill over L2 that starts from the first one's final state."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((L1 + L2, D))
    w = rng.standard_normal((ks, D))
    s0 = rng.standard_normal((1, ks - 1, D))
    y, f = oracle.short_conv_prefill(x, w, [0, L1 + L2], activation=act, initial_states=s0)
    y1, f1 = oracle.short_conv_prefill(x[:L1], w, [0, L1], activation=act, initial_states=s0)
    y2, f2 = oracle.short_conv_prefill(x[L1:], w, [0, L2], activation=act, initial_states=f1)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(f2, f)


@settings(**SETTINGS)
@given(L=st.integers(1, 10), ks=st.integers(2, 6), D=st.integers(1, 3), seed=st.integers(0, 2**16))
def test_short_conv_updates_equal_the_prefill(L, ks, D, seed):
    """L one-token updates from a conv state reproduce the prefill of those L
    tokens from the same state, outputs and final state."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((L, D))
    w = rng.standard_normal((ks, D))
    s0 = rng.standard_normal((1, ks - 1, D))
    y, f = oracle.short_conv_prefill(x, w, [0, L], initial_states=s0)
    st_ = s0
    for t in range(L):
        yt, st_ = oracle.short_conv_update(x[t:t + 1], w, st_)
        np.testing.assert_allclose(yt[0], y[t], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(st_, f)
