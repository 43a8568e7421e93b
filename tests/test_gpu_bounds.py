"""The debug build's bounds checks (libwkv7_debug.so, WKV7_DEBUG), on the GPU
without a fault.

In the debug build every plain (non-TMA) global load and store of the scan
kernels checks its address against the buffer it belongs to; an access
outside it is skipped and sets the status word (WKV7_ERR_BOUNDS from
wkv7_status). Two things are tested:

* every kernel the library selects (scalar fp32 forward and backward, the
  chunked forward and split backward for fp32 inputs, the chunked bf16
  forward, the split backward with either output pass, the fused backward,
  the fused epilogue in both directions, the no-allocation backward) runs its
  parity case through the checks with the status word
  clean and the results still equal to the oracle's: no index of theirs
  leaves its buffer;
* the checks fire: with every buffer's extent cut by 4 bytes
  (wkv7_debug_cut_extents), each call's last stores fall outside the cut
  extent, are skipped (the output's last element keeps its NaN sentinel) and
  wkv7_status reports WKV7_ERR_BOUNDS; no access leaves the real buffer. (The
  values are not compared under the cut: a skipped load of a workspace leaves
  what was there.) With the cut removed the same calls are clean again and
  write every element.
"""
import importlib.util
import os

import numpy as np
import pytest

from parity_bars import check_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")
ERR_BOUNDS = -5


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import ctypes

    import __graft_entry__  # noqa: F401
    import oracle
    from linear_rnn_state_gb300 import _build, inputs, wkv7

    _build.build()
    torch.cuda.set_device(0)
    dbg = wkv7.load(_build.DEBUG_LIB)
    dbg.wkv7_debug_cut_extents.argtypes = [ctypes.c_size_t]
    dbg.wkv7_debug_cut_extents.restype = ctypes.c_int
    dbg.wkv7_debug_out_kernel.argtypes = [ctypes.c_int]
    dbg.wkv7_debug_out_kernel.restype = ctypes.c_int
    spec = importlib.util.spec_from_file_location("epilogue_oracle", os.path.join(ROOT, "oracle", "epilogue_oracle.py"))
    epi = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(epi)
    saved = wkv7._lib
    wkv7._lib = dbg  # the torch helpers call the debug build for this module
    try:
        yield oracle, epi, inputs, wkv7, dbg
    finally:
        dbg.wkv7_debug_cut_extents(0)
        dbg.wkv7_debug_out_kernel(0)
        wkv7._lib = saved


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _data(inputs, B, T, H, N, storage, seed):
    d = dict(inputs.generate(B, T, H, N, storage, 0.1, seed=seed))
    rng = np.random.default_rng(seed + 1)
    d["dS_final"] = (0.1 * rng.standard_normal((B, H, N, N))).astype(np.float32)
    if storage == "bf16":
        t = {n: torch.from_numpy(d[n]).view(torch.bfloat16).cuda() for n in NAMES + ("dy",)}
        o = {n: inputs.as_f64(d[n], "bf16") for n in NAMES + ("dy",)}
    else:
        t = {n: torch.from_numpy(d[n]).cuda() for n in NAMES + ("dy",)}
        o = {n: d[n].astype(np.float64) for n in NAMES + ("dy",)}
    for n in ("s_init", "dS_final"):
        t[n] = torch.from_numpy(d[n].astype(np.float32)).cuda()
        o[n] = d[n].astype(np.float32).astype(np.float64)
    return t, o


def _compare(name, got, ref, bf16, kind="seq"):
    got = got.double().cpu().numpy() if hasattr(got, "cpu") else np.asarray(got, dtype=np.float64)
    if bf16:
        check_bf16(name, got, ref, kind)
    else:
        err = np.abs(got - ref) / (1.0 + np.abs(ref))
        assert err.max() <= 1e-4, f"{name}: {err.max():.3e}"


def _scan_case(env, path):
    """Forward and backward of one path through the debug build; returns the
    outputs (torch tensors) and the oracle's."""
    oracle, _, inputs, wkv7, dbg = env
    bf16 = not path.startswith("fp32")
    B, T, H, N = (2, 80, 3, 32) if path == "fp32" else (2, 130, 3, 64)
    t, o = _data(inputs, B, T, H, N, "bf16" if bf16 else "f32", seed=300 + len(path))
    dbg.wkv7_debug_out_kernel(1 if path == "tc" else 0)
    try:
        y, sf, ck, C = wkv7.forward(*(t[n] for n in NAMES), t["s_init"], ckpt_every=None if path == "fp32" else 16)
        g = wkv7.backward(*(t[n] for n in NAMES), t["dy"], t["s_init"], ck, C, dS_final=t["dS_final"],
                          fused=path == "fused")
    finally:
        dbg.wkv7_debug_out_kernel(0)
    got = {"y": y, "s_final": sf, **g}
    y_ref, sf_ref = oracle.forward(*(o[n] for n in NAMES), o["s_init"])
    gr = oracle.backward(*(o[n] for n in NAMES), o["dy"], o["s_init"], o["dS_final"])
    return got, {"y": y_ref, "s_final": sf_ref, **gr}, bf16


@pytest.mark.parametrize("path", ["fp32", "fp32-chunked", "split", "tc", "fused"])
def test_scan_kernels_stay_inside_their_buffers(env, path):
    wkv7 = env[3]
    got, ref, bf16 = _scan_case(env, path)
    assert wkv7.wkv7_status(_stream()) == 0, wkv7.last_error()
    for n, r in ref.items():
        x = got[n]
        if bf16 and n == "y":
            x = x.float()
        _compare(f"{n} ({path}, debug build)", x, r, bf16, "state" if n in ("s_final", "dS_init") else "seq")


def test_epilogue_kernels_stay_inside_their_buffers(env):
    oracle, epi, inputs, wkv7, _ = env
    B, T, H = 2, 45, 3
    t, o = _data(inputs, B, T, H, 64, "bf16", seed=331)
    rng = np.random.default_rng(5)
    ln_w = rng.uniform(0.5, 1.5, (H, 64)).astype(np.float32)
    ln_b = (0.1 * rng.standard_normal((H, 64))).astype(np.float32)
    r_k = (0.5 * rng.standard_normal((H, 64))).astype(np.float32)
    pt = [torch.from_numpy(x).cuda() for x in (ln_w, ln_b, r_k)]
    out, nv, stats, sf, ck = wkv7.forward_epilogue(*(t[n] for n in NAMES), *pt, t["s_init"])
    g = wkv7.backward_epilogue(*(t[n] for n in NAMES), t["dy"], nv, stats, pt[0], pt[2], t["s_init"], ck)
    assert wkv7.wkv7_status(_stream()) == 0, wkv7.last_error()
    y_ref, _ = oracle.forward(*(o[n] for n in NAMES), o["s_init"])
    out_ref, _ = epi.forward(y_ref, o["r"], o["k"], o["v"], ln_w, ln_b, r_k)
    _compare("out (epilogue, debug build)", out.float(), out_ref, True)
    ge = epi.backward(o["dy"], y_ref, o["r"], o["k"], o["v"], ln_w, ln_b, r_k)
    gs = oracle.backward(*(o[n] for n in NAMES), ge["dy"], o["s_init"])
    _compare("dr (epilogue, debug build)", g["dr"], gs["dr"] + ge["dr"], True)
    _compare("dw (epilogue, debug build)", g["dw"], gs["dw"], True)
    _compare("dln_w (epilogue, debug build)", g["dln_w"], ge["dln_w"], True, "state")


def test_no_alloc_backward_stays_inside_its_buffers(env):
    oracle, _, inputs, wkv7, dbg = env
    B, T, H, N = 1, 97, 3, 64
    t, o = _data(inputs, B, T, H, N, "f32", seed=333)
    g = {n: torch.empty((B, T, H, N), device="cuda") for n in GRADS}
    dS = torch.empty((B, H, N, N), device="cuda")
    rc = dbg.wkv7_backward_noalloc(*(t[n].data_ptr() for n in NAMES), t["dy"].data_ptr(), t["s_init"].data_ptr(),
                                   *(g[n].data_ptr() for n in GRADS), dS.data_ptr(), B, T, H, N, _stream())
    assert rc == 0, dbg.wkv7_last_error().decode()
    assert dbg.wkv7_status(_stream()) == 0, dbg.wkv7_last_error().decode()
    gr = oracle.backward(*(o[n] for n in NAMES), o["dy"], o["s_init"])
    for n in GRADS:
        _compare(f"{n} (no-allocation backward, debug build)", g[n], gr[n], False)


def _sentinel_run(env, path):
    """One forward and one backward of `path` into NaN-filled outputs; returns
    them and the status after each call."""
    _, _, inputs, wkv7, dbg = env
    bf16 = not path.startswith("fp32")
    B, T, H, N = (2, 80, 3, 32) if path == "fp32" else (2, 130, 3, 64)
    C = wkv7.wkv7_default_ckpt_every(N, False) if path == "fp32" else 16
    t, _ = _data(inputs, B, T, H, N, "bf16" if bf16 else "f32", seed=340)
    dev = t["r"].device
    nan = float("nan")
    y = torch.full((B, T, H, N), nan, device=dev, dtype=t["r"].dtype)
    sf = torch.full((B, H, N, N), nan, device=dev)
    ck = torch.full((B, H, (T + C - 1) // C, N, N), nan, device=dev)
    fwd = dbg.wkv7_forward_bf16 if bf16 else dbg.wkv7_forward
    rc = fwd(*(t[n].data_ptr() for n in NAMES), t["s_init"].data_ptr(), y.data_ptr(), sf.data_ptr(), ck.data_ptr(),
             C, B, T, H, N, _stream())
    assert rc == 0, dbg.wkv7_last_error().decode()
    st_fwd = dbg.wkv7_status(_stream())
    ck_out = ck.clone()
    ck.nan_to_num_(0.0)  # a checkpoint store the cut skipped must not feed NaN into the backward
    g = {n: torch.full((B, T, H, N), nan, device=dev) for n in GRADS}
    dS = torch.full((B, H, N, N), nan, device=dev)
    dbg.wkv7_debug_out_kernel(1 if path == "tc" else 0)
    try:
        fn = dbg.wkv7_backward_fused_bf16 if path == "fused" else (
            dbg.wkv7_backward_segment_bf16 if bf16 else dbg.wkv7_backward_segment)
        rc = fn(*(t[n].data_ptr() for n in NAMES), t["dy"].data_ptr(), t["s_init"].data_ptr(),
                t["dS_final"].data_ptr(), ck.data_ptr(), C, *(g[n].data_ptr() for n in GRADS), dS.data_ptr(),
                B, T, H, N, _stream())
    finally:
        dbg.wkv7_debug_out_kernel(0)
    assert rc == 0, dbg.wkv7_last_error().decode()
    st_bwd = dbg.wkv7_status(_stream())
    return {"y": y, "s_final": sf, "ckpt": ck_out, **g, "dS_init": dS}, st_fwd, st_bwd


@pytest.mark.parametrize("path", ["fp32", "fp32-chunked", "split", "tc", "fused"])
def test_a_cut_extent_is_reported_and_its_access_skipped(env, path):
    dbg = env[4]
    assert dbg.wkv7_status(_stream()) == 0
    assert dbg.wkv7_debug_cut_extents(4) == 0
    try:
        outs, st_fwd, st_bwd = _sentinel_run(env, path)
    finally:
        dbg.wkv7_debug_cut_extents(0)
    assert st_fwd == ERR_BOUNDS, (st_fwd, dbg.wkv7_last_error().decode())
    assert st_bwd == ERR_BOUNDS, (st_bwd, dbg.wkv7_last_error().decode())
    assert "outside its buffer" in dbg.wkv7_last_error().decode()
    assert dbg.wkv7_status(_stream()) == 0  # the word was cleared
    for n, x in outs.items():
        assert torch.isnan(x.float().flatten()[-1]), f"{n}: the store past the cut extent was not skipped"

    # the cut removed: the same calls are clean and write every element
    outs, st_fwd, st_bwd = _sentinel_run(env, path)
    assert st_fwd == 0 and st_bwd == 0, dbg.wkv7_last_error().decode()
    for n, x in outs.items():
        assert not torch.isnan(x.float()).any(), f"{n}: unwritten elements"
