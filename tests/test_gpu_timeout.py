"""The library's own error path for a kernel that gives up a bounded wait
(WKV7_ERR_TIMEOUT), exercised on the GPU without a fault or a hang.

The debug build (libwkv7_debug.so: 1 ms wait limit) has a hook that makes the
scalar forward issue no load for the last chunk of every head. Every CTA then
waits for a copy that was never started: after 1 ms the wait gives up, the
kernel sets the status word and every thread of the CTA leaves together.
Nothing is in flight at that point (every earlier chunk has been consumed), so
the context stays usable. The test checks that the call returns, that
wkv7_status reports WKV7_ERR_TIMEOUT once and then clears, and that a normal
forward and backward on the same device afterwards match the oracle.
"""
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__  # noqa: F401
    import ctypes

    import oracle
    from linear_rnn_state_gb300 import _build, inputs, wkv7

    _build.build()
    torch.cuda.set_device(0)
    dbg = wkv7.load(_build.DEBUG_LIB)
    dbg.wkv7_debug_skip_last_load.argtypes = [ctypes.c_int]
    dbg.wkv7_debug_skip_last_load.restype = ctypes.c_int
    yield oracle, inputs, dbg
    dbg.wkv7_debug_skip_last_load(0)


def _run(dbg, t, s0, B, T, H, N, C):
    dev = t["r"].device
    stream = torch.cuda.current_stream().cuda_stream
    y = torch.full((B, T, H, N), float("nan"), device=dev)
    sf = torch.full((B, H, N, N), float("nan"), device=dev)
    ck = torch.empty((B, H, (T + C - 1) // C, N, N), device=dev)
    rc = dbg.wkv7_forward(*(t[n].data_ptr() for n in NAMES), s0.data_ptr(), y.data_ptr(), sf.data_ptr(),
                          ck.data_ptr(), C, B, T, H, N, stream)
    return rc, y, sf, ck


def test_a_wait_that_runs_out_is_reported_and_the_device_stays_usable(env):
    oracle, inputs, dbg = env
    dev = torch.device("cuda:0")
    B, T, H, N, C = 2, 80, 3, 32, 16
    d = inputs.generate(B, T, H, N, "f32", 0.1, seed=41)
    t = {n: torch.from_numpy(d[n]).to(dev) for n in NAMES + ("dy",)}
    s0_np = d["s_init"].astype(np.float32)
    s0 = torch.from_numpy(s0_np).to(dev)
    stream = torch.cuda.current_stream().cuda_stream

    assert dbg.wkv7_status(stream) == 0, dbg.wkv7_last_error().decode()
    assert dbg.wkv7_debug_skip_last_load(1) == 0
    try:
        rc, _, _, _ = _run(dbg, t, s0, B, T, H, N, C)
        assert rc == 0, dbg.wkv7_last_error().decode()
        assert dbg.wkv7_status(stream) == -4  # WKV7_ERR_TIMEOUT
        assert "bounded wait" in dbg.wkv7_last_error().decode()
        assert dbg.wkv7_status(stream) == 0  # the word was cleared
    finally:
        dbg.wkv7_debug_skip_last_load(0)

    # the same device, the same library, a normal call: parity with the oracle
    rc, y, sf, ck = _run(dbg, t, s0, B, T, H, N, C)
    assert rc == 0
    g = {n: torch.empty((B, T, H, N), device=dev) for n in GRADS}
    dS = torch.empty((B, H, N, N), device=dev)
    rc = dbg.wkv7_backward(*(t[n].data_ptr() for n in NAMES), t["dy"].data_ptr(), s0.data_ptr(), ck.data_ptr(), C,
                           *(g[n].data_ptr() for n in GRADS), dS.data_ptr(), B, T, H, N, stream)
    assert rc == 0
    assert dbg.wkv7_status(stream) == 0
    o = {n: d[n].astype(np.float64) for n in NAMES + ("dy",)}
    y_ref, sf_ref = oracle.forward(*(o[n] for n in NAMES), s0_np.astype(np.float64))
    g_ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s0_np.astype(np.float64))
    pairs = [("y", y, y_ref), ("s_final", sf, sf_ref), ("dS_init", dS, g_ref["dS_init"])]
    pairs += [(n, g[n], g_ref[n]) for n in GRADS]
    for name, got, ref in pairs:
        got = got.double().cpu().numpy()
        err = np.abs(got - ref) / (1.0 + np.abs(ref))
        assert err.max() <= 1e-4, f"{name} after the timeout: {err.max():.3e}"
