"""libkda C ABI on the host: the library loads, exports every function that
include/kda.h declares, and rejects bad arguments before touching the GPU.
No call here launches a kernel."""
import ctypes
import os
import re

import pytest

import kimi_delta_attention_07_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kda_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    from kimi_delta_attention_07_gb300 import _build
    _build.build()
    return kda.load()


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("kda_chunk_fwd", "kda_chunk_intra", "kda_chunk_scan", "kda_recurrent_step", "kda_chunk_workspace_bytes",
              "kda_workspace_status", "kda_status_string", "kda_version", "kda_chunk_fwd_gated",
              "kda_recurrent_step_gated"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(kda.lib_path())
    for n in _declared_functions():
        assert hasattr(raw, n), f"libkda does not export {n}"
    assert set(kda.EXPORTS) <= set(_declared_functions())


def test_status_strings(lib):
    for s in range(6):
        assert kda.kda_status_string(s).startswith("KDA_")
    assert "TIMEOUT" in kda.kda_status_string(kda.KDA_ERR_DEVICE_TIMEOUT)
    assert "unknown" in kda.kda_status_string(99)
    assert lib.kda_version() == 100


def test_header_status_values_match_the_binding():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    enum = dict(re.findall(r"^\s*(KDA_(?:OK|ERR_\w+))\s*=\s*(\d+)", text, flags=re.M))
    assert {k: int(v) for k, v in enum.items()} == {
        "KDA_OK": kda.KDA_OK, "KDA_ERR_INVALID_ARG": kda.KDA_ERR_INVALID_ARG,
        "KDA_ERR_UNSUPPORTED": kda.KDA_ERR_UNSUPPORTED, "KDA_ERR_WORKSPACE": kda.KDA_ERR_WORKSPACE,
        "KDA_ERR_CUDA": kda.KDA_ERR_CUDA, "KDA_ERR_DEVICE_TIMEOUT": kda.KDA_ERR_DEVICE_TIMEOUT}
    bits = dict(re.findall(r"^#define\s+(KDA_WS_\w+)\s+(\d+)", text, flags=re.M))
    assert {k: int(v) for k, v in bits.items()} == {
        "KDA_WS_BAD_SEQLENS": kda.KDA_WS_BAD_SEQLENS, "KDA_WS_BAD_SLOT": kda.KDA_WS_BAD_SLOT,
        "KDA_WS_TIMEOUT": kda.KDA_WS_TIMEOUT, "KDA_WS_EXACT_DECAY": kda.KDA_WS_EXACT_DECAY,
        "KDA_WS_STRONG_DECAY": kda.KDA_WS_STRONG_DECAY}


@pytest.mark.parametrize("flags", range(32))
def test_workspace_status_word_maps_to_a_status(lib, flags):
    """Every combination of the status word's bits, as the kernels would leave
    them in a workspace, decodes to the documented kda_status: a bounded wait
    that gave up dominates, then the device-side argument errors; the two
    decay bits are informational."""
    st = kda.kda_status_from_workspace_flags(flags)
    if flags & kda.KDA_WS_TIMEOUT:
        assert st == kda.KDA_ERR_DEVICE_TIMEOUT
    elif flags & (kda.KDA_WS_BAD_SEQLENS | kda.KDA_WS_BAD_SLOT):
        assert st == kda.KDA_ERR_INVALID_ARG
    else:
        assert st == kda.KDA_OK
    assert kda.kda_status_string(st).startswith("KDA_")


def test_workspace_bytes(lib):
    f = kda.kda_chunk_workspace_bytes
    assert f(4096, 1, 32) > 0
    assert f(4096, 1, 32, 64, 128) == 0          # only K = V = 128 is built
    assert f(-1, 1, 32) == 0 and f(10, 0, 32) == 0 and f(10, 1, 0) == 0
    assert f(10, 1, 32, dtype=7) == 0
    # grows with tokens, sequences and heads; covers one record per (chunk, head)
    assert f(8192, 1, 32) > f(4096, 1, 32)
    assert f(4096, 4, 32) > f(4096, 1, 32)
    assert f(4096, 1, 32) >= (4096 // 64) * 32 * 64 * 128 * 2


def _chunk(lib, **kw):
    a = dict(q=8, k=8, v=8, g=16, beta=16, s0=None, sf=None, idx=None, slots=0, o=8, cu=None,
             N=1, T=64, H=1, K=128, V=128, scale=0.1, dt=kda.KDA_BF16, flags=0, ws=256,
             wsb=1 << 30, stream=None)
    a.update(kw)
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.kda_chunk_fwd(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["g"]), vp(a["beta"]),
                             vp(a["s0"]), vp(a["sf"]), vp(a["idx"]), a["slots"], vp(a["o"]),
                             vp(a["cu"]), a["N"], a["T"], a["H"], a["K"], a["V"], a["scale"],
                             a["dt"], a["flags"], vp(a["ws"]), a["wsb"], None)


def test_chunk_fwd_rejects_bad_arguments_without_launching(lib):
    # fake, never-dereferenced addresses: validation fails before any launch
    base = 1 << 20
    ok = dict(q=base, k=base, v=base, g=base, beta=base, o=base, ws=base)
    assert _chunk(lib, **{**ok, "dt": 5}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, **{**ok, "K": 64}) == kda.KDA_ERR_UNSUPPORTED
    assert _chunk(lib, **{**ok, "q": None}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, **{**ok, "N": 0}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, **{**ok, "T": -1}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, **{**ok, "N": 3, "T": 64}) == kda.KDA_ERR_INVALID_ARG  # 3 does not divide 64
    assert _chunk(lib, **{**ok, "flags": 16}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, **{**ok, "flags": kda.KDA_CHUNK_SCAN_WIDE | kda.KDA_CHUNK_SCAN_SPLIT}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, **{**ok, "q": base + 2}) == kda.KDA_ERR_INVALID_ARG   # misaligned row
    assert _chunk(lib, **{**ok, "ws": None}) == kda.KDA_ERR_WORKSPACE
    assert _chunk(lib, **{**ok, "ws": base + 16}) == kda.KDA_ERR_WORKSPACE   # not 256-aligned
    assert _chunk(lib, **{**ok, "wsb": 1024}) == kda.KDA_ERR_WORKSPACE
    assert _chunk(lib, **{**ok, "idx": base, "slots": 0}) == kda.KDA_ERR_INVALID_ARG
    assert _chunk(lib, **{**ok, "scale": float("nan")}) == kda.KDA_ERR_INVALID_ARG


def test_gated_entry_points_reject_bad_arguments_without_launching(lib):
    base = 1 << 20
    vp = ctypes.c_void_p
    p = lambda x: None if x is None else vp(x)

    def chunk(**kw):
        a = dict(q=base, k=base, v=base, rg=base, rb=base, alog=base, bias=base, lb=-5.0, use_lb=1,
                 og=None, nw=base, eps=1e-6, o=base, N=1, T=64, H=1, dt=kda.KDA_BF16, flags=0,
                 ws=base, wsb=1 << 30)
        a.update(kw)
        return lib.kda_chunk_fwd_gated(p(a["q"]), p(a["k"]), p(a["v"]), p(a["rg"]), p(a["rb"]),
                                       p(a["alog"]), p(a["bias"]), a["lb"], a["use_lb"], p(a["og"]),
                                       p(a["nw"]), a["eps"], None, None, None, 0, p(a["o"]), None,
                                       a["N"], a["T"], a["H"], 128, 128, 0.1, a["dt"], a["flags"],
                                       p(a["ws"]), a["wsb"], None)

    def step(**kw):
        a = dict(q=base, k=base, v=base, rg=base, rb=base, alog=base, bias=base, lb=-5.0, use_lb=1,
                 og=None, nw=base, eps=1e-6, pool=base, o=base, N=2, H=2, dt=kda.KDA_F32)
        a.update(kw)
        return lib.kda_recurrent_step_gated(p(a["q"]), p(a["k"]), p(a["v"]), p(a["rg"]), p(a["rb"]),
                                            p(a["alog"]), p(a["bias"]), a["lb"], a["use_lb"],
                                            p(a["og"]), p(a["nw"]), a["eps"], p(a["pool"]), None, 4,
                                            p(a["o"]), a["N"], a["H"], 128, 128, 0.1, a["dt"], None)

    for f in (chunk, step):
        assert f(alog=None) == kda.KDA_ERR_INVALID_ARG
        assert f(bias=None) == kda.KDA_ERR_INVALID_ARG
        assert f(bias=base + 4) == kda.KDA_ERR_INVALID_ARG      # dt_bias rows: 16-byte aligned
        assert f(rg=None) == kda.KDA_ERR_INVALID_ARG
        assert f(rb=None) == kda.KDA_ERR_INVALID_ARG
        assert f(lb=float("nan")) == kda.KDA_ERR_INVALID_ARG    # a lower bound must be finite
        assert f(dt=4) == kda.KDA_ERR_INVALID_ARG
        # output epilogue: weight needed, 16-byte aligned, positive finite eps
        assert f(og=base, nw=None) == kda.KDA_ERR_INVALID_ARG
        assert f(og=base, nw=base + 4) == kda.KDA_ERR_INVALID_ARG
        assert f(og=base, eps=0.0) == kda.KDA_ERR_INVALID_ARG
        assert f(og=base, eps=float("inf")) == kda.KDA_ERR_INVALID_ARG
    assert chunk(rg=base + 8) == kda.KDA_ERR_INVALID_ARG        # tensor-core path: 16-byte rows
    assert chunk(ws=None) == kda.KDA_ERR_WORKSPACE
    # the fp32 path keeps the activated gate in the workspace: it needs more room
    f32 = kda.kda_chunk_workspace_bytes(4096, 1, 32, dtype=kda.KDA_F32)
    f32_gated = kda.kda_chunk_workspace_bytes(4096, 1, 32, dtype=kda.KDA_F32, flags=kda.KDA_CHUNK_GATED)
    assert f32_gated >= f32 + 4096 * 32 * (128 + 1) * 4
    assert (kda.kda_chunk_workspace_bytes(4096, 1, 32, flags=kda.KDA_CHUNK_GATED)
            == kda.kda_chunk_workspace_bytes(4096, 1, 32))          # tensor-core path: on chip


def test_output_gate_norm_rejects_bad_arguments_without_launching(lib):
    base = 1 << 20
    vp = ctypes.c_void_p
    f = lambda o=base, g=base, w=base, eps=1e-6, rows=10, V=128, dt=kda.KDA_BF16: \
        lib.kda_output_gate_norm(None if o is None else vp(o), None if g is None else vp(g),
                                 None if w is None else vp(w), eps, rows, V, dt, None)
    assert f(rows=0) == kda.KDA_OK                      # nothing to do
    assert f(V=64) == kda.KDA_ERR_UNSUPPORTED
    assert f(rows=-1) == kda.KDA_ERR_INVALID_ARG
    assert f(o=None) == kda.KDA_ERR_INVALID_ARG
    assert f(g=None) == kda.KDA_ERR_INVALID_ARG
    assert f(w=None) == kda.KDA_ERR_INVALID_ARG
    assert f(w=base + 8) == kda.KDA_ERR_INVALID_ARG
    assert f(eps=-1.0) == kda.KDA_ERR_INVALID_ARG
    assert f(o=base + 4) == kda.KDA_ERR_INVALID_ARG      # bf16 rows: 8-byte aligned
    assert f(dt=kda.KDA_F32, g=base + 8) == kda.KDA_ERR_INVALID_ARG


def test_multi_step_rejects_bad_arguments_without_launching(lib):
    base = 1 << 20
    vp = ctypes.c_void_p
    p = lambda x: None if x is None else vp(x)

    def f(**kw):
        a = dict(q=base, k=base, v=base, g=base, b=base, pool=base, idx=base, acc=None, slots=8,
                 o=base, N=2, S=3, H=2, dt=kda.KDA_BF16)
        a.update(kw)
        return lib.kda_recurrent_multi_step(p(a["q"]), p(a["k"]), p(a["v"]), p(a["g"]), p(a["b"]),
                                            p(a["pool"]), p(a["idx"]), p(a["acc"]), a["slots"],
                                            p(a["o"]), a["N"], a["S"], a["H"], 128, 128, 0.1, a["dt"],
                                            None)

    assert f(N=0) == kda.KDA_OK
    assert f(S=0) == kda.KDA_ERR_INVALID_ARG
    assert f(idx=None) == kda.KDA_ERR_INVALID_ARG       # per-token slots are required for S > 1
    assert f(pool=None) == kda.KDA_ERR_INVALID_ARG
    assert f(g=base + 4) == kda.KDA_ERR_INVALID_ARG
    assert f(dt=2) == kda.KDA_ERR_INVALID_ARG

    def fg(**kw):  # the gated form: raw gates, gate parameters, optional epilogue
        a = dict(q=base, k=base, v=base, rg=base, rb=base, alog=base, bias=base, lb=-5.0, og=None,
                 nw=None, eps=1e-6, pool=base, idx=base, acc=None, slots=8, o=base, N=2, S=3, H=2,
                 dt=kda.KDA_BF16)
        a.update(kw)
        return lib.kda_recurrent_multi_step_gated(
            p(a["q"]), p(a["k"]), p(a["v"]), p(a["rg"]), p(a["rb"]), p(a["alog"]), p(a["bias"]),
            a["lb"], 1, p(a["og"]), p(a["nw"]), a["eps"], p(a["pool"]), p(a["idx"]), p(a["acc"]),
            a["slots"], p(a["o"]), a["N"], a["S"], a["H"], 128, 128, 0.1, a["dt"], None)

    assert fg(N=0) == kda.KDA_OK
    assert fg(S=0) == kda.KDA_ERR_INVALID_ARG
    assert fg(idx=None) == kda.KDA_ERR_INVALID_ARG
    assert fg(rg=None) == kda.KDA_ERR_INVALID_ARG
    assert fg(alog=None) == kda.KDA_ERR_INVALID_ARG
    assert fg(og=base, nw=None) == kda.KDA_ERR_INVALID_ARG   # an epilogue needs its weight
    assert fg(og=base, nw=base, eps=0.0) == kda.KDA_ERR_INVALID_ARG


def test_short_conv_rejects_bad_arguments_without_launching(lib):
    base = 1 << 20
    vp = ctypes.c_void_p
    p = lambda x: None if x is None else vp(x)

    def fwd(**kw):
        a = dict(x=base, w=base, y=base, cu=None, N=1, T=64, D=256, ks=4, act=1, s0=None, sf=None,
                 idx=None, slots=0, dt=kda.KDA_BF16)
        a.update(kw)
        return lib.kda_short_conv_fwd(p(a["x"]), p(a["w"]), p(a["y"]), p(a["cu"]), a["N"], a["T"],
                                      a["D"], a["ks"], a["act"], p(a["s0"]), p(a["sf"]), p(a["idx"]),
                                      a["slots"], a["dt"], None)

    def upd(**kw):
        a = dict(x=base, w=base, y=base, pool=base, idx=None, slots=4, N=4, D=256, ks=4, act=1,
                 dt=kda.KDA_BF16)
        a.update(kw)
        return lib.kda_short_conv_update(p(a["x"]), p(a["w"]), p(a["y"]), p(a["pool"]), p(a["idx"]),
                                         a["slots"], a["N"], a["D"], a["ks"], a["act"], a["dt"], None)

    for f in (fwd, upd):
        assert f(ks=1) == kda.KDA_ERR_INVALID_ARG
        assert f(ks=9) == kda.KDA_ERR_INVALID_ARG
        assert f(D=100) == kda.KDA_ERR_INVALID_ARG      # D a multiple of 8
        assert f(act=2) == kda.KDA_ERR_INVALID_ARG
        assert f(dt=3) == kda.KDA_ERR_INVALID_ARG
        assert f(x=None) == kda.KDA_ERR_INVALID_ARG
        assert f(x=base + 8) == kda.KDA_ERR_INVALID_ARG  # bf16 rows of 8 channels: 16 bytes
    assert fwd(N=3, T=64) == kda.KDA_ERR_INVALID_ARG     # 3 does not divide 64
    assert fwd(idx=base, slots=0) == kda.KDA_ERR_INVALID_ARG
    assert upd(N=0) == kda.KDA_OK
    assert upd(slots=3) == kda.KDA_ERR_INVALID_ARG       # identity slots need slots >= N
    assert upd(pool=None) == kda.KDA_ERR_INVALID_ARG


    def multi(**kw):
        a = dict(x=base, w=base, y=base, pool=base, idx=base, acc=None, slots=16, N=4, S=4, D=256,
                 ks=4, act=1, dt=kda.KDA_BF16)
        a.update(kw)
        return lib.kda_short_conv_multi_update(p(a["x"]), p(a["w"]), p(a["y"]), p(a["pool"]),
                                               p(a["idx"]), p(a["acc"]), a["slots"], a["N"], a["S"],
                                               a["D"], a["ks"], a["act"], a["dt"], None)

    assert multi(N=0) == kda.KDA_OK
    for bad in (dict(S=0), dict(idx=None), dict(slots=0), dict(ks=9), dict(D=12), dict(act=5),
                dict(dt=7), dict(y=base + 4), dict(pool=None)):
        assert multi(**bad) == kda.KDA_ERR_INVALID_ARG, bad


def test_recurrent_step_rejects_bad_arguments_without_launching(lib):
    base = 1 << 20
    vp = ctypes.c_void_p

    def step(**kw):
        a = dict(q=base, k=base, v=base, g=base, beta=base, pool=base, idx=None, slots=4, o=base,
                 N=4, H=2, K=128, V=128, scale=0.1, dt=kda.KDA_F32)
        a.update(kw)
        p = lambda x: None if x is None else vp(x)
        return lib.kda_recurrent_step(p(a["q"]), p(a["k"]), p(a["v"]), p(a["g"]), p(a["beta"]),
                                      p(a["pool"]), p(a["idx"]), a["slots"], p(a["o"]), a["N"],
                                      a["H"], a["K"], a["V"], a["scale"], a["dt"], None)

    assert step(N=0) == kda.KDA_OK                         # empty batch: nothing to do
    assert step(V=64) == kda.KDA_ERR_UNSUPPORTED
    assert step(pool=None) == kda.KDA_ERR_INVALID_ARG
    assert step(slots=3) == kda.KDA_ERR_INVALID_ARG         # identity slots need slots >= N
    assert step(N=-1) == kda.KDA_ERR_INVALID_ARG
    assert step(dt=3) == kda.KDA_ERR_INVALID_ARG
    assert step(g=base + 4) == kda.KDA_ERR_INVALID_ARG      # g rows must be 16-byte aligned


def test_product_path_does_not_touch_the_oracle():
    # the library package and its sources never import or name the oracle
    pkg = os.path.join(ROOT, "kimi_delta_attention_07_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "kda_oracle" not in text, fn
