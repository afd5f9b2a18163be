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
import numpy as np
import pytest
import torch

import kda_inputs

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 1e-2


@pytest.fixture(scope="module")
def kda():
    import kimi_delta_attention_07_gb300 as m
    m.load()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    return m


def rel_l2(x, ref):
    x = x.detach().double().cpu().numpy()
    ref = ref.detach().double().cpu().numpy()
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


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
    # first call: fp32, ragged packed sequences (one empty), nonzero initial state
    x1 = kda_inputs.prefill([200, 77, 0, 64], H=4, dtype=torch.float32, seed=41, init_std=0.02)
    o, s, o_ref, s_ref = _both(kda, x1)
    assert rel_l2(o, o_ref) < TOL_F32
    assert rel_l2(s, s_ref) < TOL_F32
    # second call right after, other sizes and dtype: the shared scratch array
    # holds the first call's data and must not leak into this one
    x2 = kda_inputs.prefill([130, 5], H=3, dtype=torch.bfloat16, seed=42)
    o, s, o_ref, s_ref = _both(kda, x2)
    assert rel_l2(o, o_ref) < TOL_BF16
    assert rel_l2(s, s_ref) < TOL_BF16
    assert torch.isfinite(o).all() and torch.isfinite(s).all()


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
