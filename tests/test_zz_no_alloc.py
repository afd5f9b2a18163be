"""kda_chunk_fwd_noalloc against kda_chunk_fwd.

The no-alloc entry point exists for hosts that cannot allocate device memory
(a server plugin that only receives its input and output buffers, or a
latency-critical path where cudaMalloc may synchronise the device).  It
must give the same results as the regular entry point, which takes a
caller-allocated workspace, on consecutive calls that share its fixed
scratch array, and must refuse sizes its array cannot hold.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test.
"""
import pytest
import torch

import kda_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    import kimi_delta_attention_07_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return m


def _both(kda, x, precise=False):
    d = {n: (x[n].cuda() if x[n] is not None else None)
         for n in ("q", "k", "v", "g", "beta", "cu_seqlens", "initial_state")}
    T, H, _ = x["q"].shape
    N = len(x["lengths"])
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
    kw = dict(cu_seqlens=d["cu_seqlens"], initial_state=d["initial_state"], precise=precise)
    o_ref, s_ref = kda.kda_chunk_fwd(*args, **kw)
    o = torch.empty_like(o_ref)
    s = torch.empty((N, H, 128, 128), dtype=torch.float32, device="cuda")
    kda.kda_chunk_fwd_noalloc(*args, o=o, final_state=s, **kw)
    torch.cuda.synchronize()
    return o, s, o_ref, s_ref


def test_noalloc_matches_workspace_entry_point_on_two_calls(kda):
    # Both entry points run the same kernels on the same inputs with the same
    # launch shapes, so their results agree bit for bit.
    # first call: fp32, ragged packed sequences (one empty), nonzero initial state
    x1 = kda_inputs.prefill([200, 77, 0, 64], H=4, dtype=torch.float32, seed=41, init_std=0.02)
    o, s, o_ref, s_ref = _both(kda, x1)
    assert torch.equal(o, o_ref) and torch.equal(s, s_ref)
    # second call right after, other sizes and dtype: the shared scratch array
    # holds the first call's data and must not leak into this one
    x2 = kda_inputs.prefill([130, 5], H=3, dtype=torch.bfloat16, seed=42)
    o, s, o_ref, s_ref = _both(kda, x2)
    assert torch.equal(o, o_ref) and torch.equal(s, s_ref)
    assert torch.isfinite(o).all() and torch.isfinite(s).all()


def test_noalloc_hands_states_into_a_pool_in_place(kda):
    """Slot pool with state_indices, final_state the same tensor as
    initial_state (the prefill-to-decode hand-off done in place), against
    kda_chunk_fwd on a copy of the same pool."""
    x = kda_inputs.prefill([150, 64, 9], H=2, dtype=torch.bfloat16, seed=43)
    d = {n: x[n].cuda() for n in ("q", "k", "v", "g", "beta", "cu_seqlens")}
    pool = kda_inputs.decode_pool(6, H=2, seed=43).cuda()
    idx = torch.tensor([4, 0, 2], dtype=torch.int32, device="cuda")
    pool_ref, pool_na = pool.clone(), pool.clone()
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
    o_ref, _ = kda.kda_chunk_fwd(*args, cu_seqlens=d["cu_seqlens"], initial_state=pool_ref,
                                 final_state=pool_ref, state_indices=idx)
    o = torch.empty_like(o_ref)
    kda.kda_chunk_fwd_noalloc(*args, o=o, cu_seqlens=d["cu_seqlens"], initial_state=pool_na,
                              final_state=pool_na, state_indices=idx)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(pool_na, pool_ref)
    assert torch.equal(pool_na[[1, 3, 5]], pool[[1, 3, 5]])  # untouched slots
    assert not torch.equal(pool_na[4], pool[4])


def test_noalloc_wrapper_checks_arguments_like_the_workspace_entry_point(kda):
    x = kda_inputs.prefill([70], H=2, dtype=torch.bfloat16, seed=44)
    d = {n: x[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    o = torch.empty((70, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):  # g must be fp32
        kda.kda_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"].bfloat16(), d["beta"], o=o)
    with pytest.raises(ValueError):  # o too short
        kda.kda_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], o=o[:60])
    idx = torch.tensor([3], dtype=torch.int32, device="cuda")
    pool = torch.zeros((4, 2, 128, 128), device="cuda")
    with pytest.raises(ValueError):  # a pool needs a destination
        kda.kda_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], o=o,
                                  initial_state=pool, state_indices=idx)
    with pytest.raises(ValueError):  # initial pool smaller than n_slots
        kda.kda_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], o=o,
                                  initial_state=pool[:2], final_state=pool, state_indices=idx)


def test_noalloc_refuses_sizes_beyond_its_array(kda):
    H, T = 32, 4096  # needs far more than the fixed 64 MiB
    assert kda.kda_chunk_workspace_bytes(T, 1, H) > kda.NOALLOC_WORKSPACE_BYTES
    z = torch.zeros((T, H, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((T, H, 128), dtype=torch.float32, device="cuda")
    b = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    o = torch.full((T, H, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    s = torch.full((1, H, 128, 128), 5.0, device="cuda")
    with pytest.raises(kda.KdaError) as err:
        kda.kda_chunk_fwd_noalloc(z, z, z, g, b, o=o, final_state=s)
    assert err.value.status == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (o == 3.0).all() and (s == 5.0).all()  # nothing was enqueued
