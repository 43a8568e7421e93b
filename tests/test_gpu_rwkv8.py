"""GPU parity of the RWKV-8 normalized recurrence (include/rwkv8.h) against the
fp64 oracle (oracle/rwkv8_oracle.py), called through the C ABI.

Inputs are the seeded synthetic ones of linear_rnn_state_gb300.inputs
(generate_rwkv8), rounded to fp32; the oracle consumes exactly those values.
Every launch form is checked: by default the forward's chain between chunks
runs alone and its per-chunk work for all chunks at once, and the backward
walks each (b, h) through its chunks in one CTA; RWKV8_SEQUENTIAL=1 walks each
(b, h) through its chunks in the forward too; RWKV8_SPLIT_BACKWARD=1 runs the
backward's carried gradients alone and then every chunk at once.
The bar is the fp32 one of this library, element by element:
|gpu - ref| <= 1e-4 (1 + |ref|) for y, the final states, dq, dv and the
initial-state gradients. ddecay is a sum over batch and time of terms of both
signs, so one entry can be much smaller than the terms it sums; it is held to
|gpu - ref| <= 1e-4 (1 + |ref| + S) with S the mean |ref| over its latents
(the scale of the summands, which fp32 summation error follows).
"""
import importlib.util
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__  # noqa: F401
    from linear_rnn_state_gb300 import _build, inputs, rwkv8

    _build.build()
    rwkv8.load()
    spec = importlib.util.spec_from_file_location("rwkv8_oracle", os.path.join(ROOT, "oracle", "rwkv8_oracle.py"))
    orc = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(orc)
    torch.cuda.set_device(0)
    return orc, inputs, rwkv8


def _close(name, got, ref, scale=0.0):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), name
    err = np.abs(got - ref) / (1.0 + np.abs(ref) + scale)
    assert err.max() <= 1e-4, f"{name}: max scaled error {err.max():.3e}"


def _dq_rounding_scale(o):
    """Per element of dq, the fp32 rounding allowance of its first term, in
    the units of _close's `scale`. dq_t = (g_qw - <g_qw, qw>) / (sum q_t + EPS)
    + ..., g_qw[l] = R / (n_t[l] + EPS), R = sum_e rho_t[l][e] dy_t[e]: on a
    query row of zeros the sum q_t is 0, so the signed 64-term sum R is divided
    by EPS = 1e-6, and where R cancels to a small fraction of its terms no fp32
    evaluation of it (in any order) holds 1e-4 of the result. The allowance is
    the standard bound for a sum of 64 products, 64 * 2^-24 * sum_e |rho dy|,
    carried through the two divisions; added, as for ddecay, to the bar's scale
    (1e-4 (1 + |ref| + scale)). Away from such rows it is a few 1e-2 of the bar.
    States from the recurrence rho <- d rho + q v^T, n <- d n + q (state before
    each step)."""
    q, v, dy, dec = o["q"], o["v"], o["dy"], o["decay"]
    B, H, T, L = q.shape
    Hv = v.shape[1]
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            rho = np.zeros((L, v.shape[3])) if o["rho_init"] is None else o["rho_init"][b, h].copy()
            n = np.zeros(L) if o["rho_norm_init"] is None else o["rho_norm_init"][b, h].copy()
            vv = v[b, 0 if Hv == 1 else h]
            for t in range(T):
                terms = np.abs(rho * dy[b, h, t][None, :]).sum(axis=1)
                out[b, h, t] = 64 * 2.0 ** -24 * terms / ((n + 1e-6) * (q[b, h, t].sum() + 1e-6)) / 1e-4
                rho = dec[h][:, None] * rho + np.outer(q[b, h, t], vv[t])
                n = dec[h] * n + q[b, h, t]
    return out


def _dev(x):
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _run(env, B, T, H, Hv, seed, state=False, boundary=False, use_ckpt=True):
    orc, inputs, rwkv8 = env
    d = inputs.generate_rwkv8(B, T, H, Hv, 64, 64, "f32", state_std=0.1 if state else None, boundary=boundary,
                              seed=seed)
    t = {k: _dev(x) for k, x in d.items()}
    y, rf, nf, ck = rwkv8.forward(t["q"], t["v"], t["decay"], t["rho_init"], t["rho_norm_init"], want_ckpt=use_ckpt)
    g = rwkv8.backward(t["q"], t["v"], t["decay"], t["dy"], t["rho_init"], t["rho_norm_init"], ck,
                       d_rho_final=t["d_rho_final"], d_rho_norm_final=t["d_rho_norm_final"])
    torch.cuda.synchronize()
    o = {k: None if x is None else x.astype(np.float64) for k, x in d.items()}
    y_ref, rf_ref, nf_ref = orc.forward(o["q"], o["v"], o["decay"], o["rho_init"], o["rho_norm_init"])
    g_ref = orc.backward(o["q"], o["v"], o["decay"], o["dy"], o["rho_init"], o["rho_norm_init"], o["d_rho_final"],
                         o["d_rho_norm_final"])
    tag = f"B={B} T={T} H={H} Hv={Hv}"
    _close(f"y {tag}", y.cpu().numpy(), y_ref)
    _close(f"rho_final {tag}", rf.cpu().numpy(), rf_ref)
    _close(f"rho_norm_final {tag}", nf.cpu().numpy(), nf_ref)
    for k in ("dq", "dv", "d_rho_init", "d_rho_norm_init"):
        _close(f"{k} {tag}", g[k].cpu().numpy(), g_ref[k])
    _close(f"ddecay {tag}", g["ddecay"].cpu().numpy(), g_ref["ddecay"], float(np.abs(g_ref["ddecay"]).mean()))
    return g


VARIANTS = ["chunked", "sequential", "split_backward"]


def _variant(monkeypatch, variant):
    monkeypatch.delenv("RWKV8_SEQUENTIAL", raising=False)
    monkeypatch.delenv("RWKV8_SPLIT_BACKWARD", raising=False)
    if variant == "sequential":
        monkeypatch.setenv("RWKV8_SEQUENTIAL", "1")
    elif variant == "split_backward":
        monkeypatch.setenv("RWKV8_SPLIT_BACKWARD", "1")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("B,T,H,Hv", [(2, 16, 3, 3), (2, 45, 3, 1), (1, 130, 2, 2), (2, 1, 2, 2), (1, 33, 1, 1)])
def test_rwkv8_parity(env, B, T, H, Hv, variant, monkeypatch):
    _variant(monkeypatch, variant)
    _run(env, B, T, H, Hv, seed=100 + T)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("Hv", [1, 3])
def test_rwkv8_parity_with_states_and_boundary(env, Hv, variant, monkeypatch):
    _variant(monkeypatch, variant)
    _run(env, 2, 70, 3, Hv, seed=7, state=True, boundary=True)
    _run(env, 1, 70, 3, Hv, seed=8, state=True, boundary=True, use_ckpt=False)


def test_rwkv8_backward_without_checkpoints_matches(env):
    """ckpt = NULL makes the library run the forward itself: the same kernels
    on the same inputs, so the gradients are bit-identical."""
    _, inputs, rwkv8 = env
    d = inputs.generate_rwkv8(2, 50, 2, 2, 64, 64, "f32", state_std=0.1, seed=3)
    t = {k: _dev(x) for k, x in d.items()}
    _, _, _, ck = rwkv8.forward(t["q"], t["v"], t["decay"], t["rho_init"], t["rho_norm_init"])
    g1 = rwkv8.backward(t["q"], t["v"], t["decay"], t["dy"], t["rho_init"], t["rho_norm_init"], ck)
    g2 = rwkv8.backward(t["q"], t["v"], t["decay"], t["dy"], t["rho_init"], t["rho_norm_init"], None)
    torch.cuda.synchronize()
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_rwkv8_empty_sequence(env):
    _, inputs, rwkv8 = env
    d = inputs.generate_rwkv8(2, 1, 2, 2, 64, 64, "f32", state_std=0.1, boundary=True, seed=4)
    t = {k: _dev(x) for k, x in d.items()}
    q0, v0, dy0 = (torch.empty((2, 2, 0, 64), device="cuda") for _ in range(3))
    y, rf, nf, _ = rwkv8.forward(q0, v0, t["decay"], t["rho_init"], t["rho_norm_init"], want_ckpt=False)
    g = rwkv8.backward(q0, v0, t["decay"], dy0, t["rho_init"], t["rho_norm_init"], None,
                       d_rho_final=t["d_rho_final"], d_rho_norm_final=t["d_rho_norm_final"])
    torch.cuda.synchronize()
    assert torch.equal(rf, t["rho_init"]) and torch.equal(nf, t["rho_norm_init"])
    assert torch.equal(g["d_rho_init"], t["d_rho_final"]) and torch.equal(g["d_rho_norm_init"], t["d_rho_norm_final"])
    assert torch.count_nonzero(g["ddecay"]) == 0


def test_rwkv8_segments_compose(env):
    """Backward of [T1, T) with the final-state gradients, then of [0, T1) with
    the initial-state gradients it returned, equals the whole sequence's."""
    _, inputs, rwkv8 = env
    B, T, H, T1 = 2, 96, 2, 40
    d = inputs.generate_rwkv8(B, T, H, H, 64, 64, "f32", boundary=True, seed=5)
    t = {k: _dev(x) for k, x in d.items()}
    full = rwkv8.backward(t["q"], t["v"], t["decay"], t["dy"], None, None, None, d_rho_final=t["d_rho_final"],
                          d_rho_norm_final=t["d_rho_norm_final"])
    a = {k: t[k][:, :, :T1].contiguous() for k in ("q", "v", "dy")}
    z = {k: t[k][:, :, T1:].contiguous() for k in ("q", "v", "dy")}
    _, r_mid, n_mid, _ = rwkv8.forward(a["q"], a["v"], t["decay"], want_ckpt=False)
    g2 = rwkv8.backward(z["q"], z["v"], t["decay"], z["dy"], r_mid, n_mid, None, d_rho_final=t["d_rho_final"],
                        d_rho_norm_final=t["d_rho_norm_final"])
    g1 = rwkv8.backward(a["q"], a["v"], t["decay"], a["dy"], None, None, None, d_rho_final=g2["d_rho_init"],
                        d_rho_norm_final=g2["d_rho_norm_init"])
    torch.cuda.synchronize()
    for k in ("dq", "dv"):
        got = torch.cat([g1[k], g2[k]], dim=2).cpu().numpy()
        _close(k, got, full[k].cpu().numpy().astype(np.float64))
    _close("ddecay", (g1["ddecay"] + g2["ddecay"]).cpu().numpy(), full["ddecay"].cpu().numpy().astype(np.float64),
           float(np.abs(full["ddecay"].cpu().numpy()).mean()))


def test_rwkv8_full_size_sampled(env):
    """The benchmark's workload (B=4, T=4096, H=32, one value row per head,
    L = E = 64) in the same launch configuration; the oracle recomputes every
    output of the heads of one h (all four batch rows, so ddecay[h] is whole)."""
    orc, inputs, rwkv8 = env
    B, T, H = 4, 4096, 32
    d = inputs.generate_rwkv8(B, T, H, H, 64, 64, "f32", seed=0)
    t = {k: _dev(x) for k, x in d.items()}
    y, rf, nf, ck = rwkv8.forward(t["q"], t["v"], t["decay"])
    g = rwkv8.backward(t["q"], t["v"], t["decay"], t["dy"], None, None, ck)
    torch.cuda.synchronize()
    for h in (0, 31):
        sl = (slice(None), slice(h, h + 1))
        o = {k: d[k][sl].astype(np.float64) for k in ("q", "v", "dy")}
        dec = d["decay"][h:h + 1].astype(np.float64)
        y_ref, rf_ref, nf_ref = orc.forward(o["q"], o["v"], dec)
        g_ref = orc.backward(o["q"], o["v"], dec, o["dy"])
        _close(f"y h={h}", y[sl].cpu().numpy(), y_ref)
        _close(f"rho_final h={h}", rf[sl].cpu().numpy(), rf_ref)
        _close(f"rho_norm_final h={h}", nf[sl].cpu().numpy(), nf_ref)
        for k in ("dq", "dv", "d_rho_init", "d_rho_norm_init"):
            _close(f"{k} h={h}", g[k][sl].cpu().numpy(), g_ref[k])
        _close(f"ddecay h={h}", g["ddecay"][h:h + 1].cpu().numpy(), g_ref["ddecay"],
               float(np.abs(g_ref["ddecay"]).mean()))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("case", ["decay_zero", "decay_one", "zero_query_rows", "mixed_decay"])
def test_rwkv8_degenerate_inputs(env, case, variant, monkeypatch):
    """Decay exactly 0 (only the previous step is seen) or 1 (plain prefix
    sums), query rows of zeros (their weights are 0 / EPS = 0), and a decay
    that mixes 0, 1 and tiny values across latents. dq carries the rounding
    allowance of _dq_rounding_scale: on the rows of zeros it divides a signed
    sum by EPS."""
    _variant(monkeypatch, variant)
    orc, inputs, rwkv8 = env
    B, T, H = 2, 40, 2
    d = inputs.generate_rwkv8(B, T, H, H, 64, 64, "f32", state_std=0.1, boundary=True, seed=90)
    if case == "decay_zero":
        d["decay"][:] = 0.0
    elif case == "decay_one":
        d["decay"][:] = 1.0
    elif case == "zero_query_rows":
        d["q"][:, :, 5:9, :] = 0.0
        d["q"][:, :, 20, :] = 0.0
    else:
        d["decay"][:, 0::3] = 0.0
        d["decay"][:, 1::3] = 1.0
        d["decay"][:, 2::6] = 1e-30
    t = {k: _dev(x) for k, x in d.items()}
    y, rf, nf, ck = rwkv8.forward(t["q"], t["v"], t["decay"], t["rho_init"], t["rho_norm_init"])
    g = rwkv8.backward(t["q"], t["v"], t["decay"], t["dy"], t["rho_init"], t["rho_norm_init"], ck,
                       d_rho_final=t["d_rho_final"], d_rho_norm_final=t["d_rho_norm_final"])
    torch.cuda.synchronize()
    o = {k: None if x is None else x.astype(np.float64) for k, x in d.items()}
    y_ref, rf_ref, nf_ref = orc.forward(o["q"], o["v"], o["decay"], o["rho_init"], o["rho_norm_init"])
    g_ref = orc.backward(o["q"], o["v"], o["decay"], o["dy"], o["rho_init"], o["rho_norm_init"], o["d_rho_final"],
                         o["d_rho_norm_final"])
    _close(f"y {case}", y.cpu().numpy(), y_ref)
    _close(f"rho_final {case}", rf.cpu().numpy(), rf_ref)
    _close(f"rho_norm_final {case}", nf.cpu().numpy(), nf_ref)
    _close(f"dq {case}", g["dq"].cpu().numpy(), g_ref["dq"], _dq_rounding_scale(o))
    for k in ("dv", "d_rho_init", "d_rho_norm_init"):
        _close(f"{k} {case}", g[k].cpu().numpy(), g_ref[k])
    _close(f"ddecay {case}", g["ddecay"].cpu().numpy(), g_ref["ddecay"], float(np.abs(g_ref["ddecay"]).mean()))


def test_rwkv8_launch_forms_agree(env, monkeypatch):
    """The launch forms on one input of several chunks and a ragged tail: the
    forward's y, final states and checkpoints, and every gradient, agree to
    fp32 rounding (the chains sum their terms in another order)."""
    _, inputs, rwkv8 = env
    d = inputs.generate_rwkv8(2, 77, 3, 3, 64, 64, "f32", state_std=0.1, boundary=True, seed=12)
    t = {k: _dev(x) for k, x in d.items()}
    out = {}
    for variant in VARIANTS:
        _variant(monkeypatch, variant)
        f = rwkv8.forward(t["q"], t["v"], t["decay"], t["rho_init"], t["rho_norm_init"])
        g = rwkv8.backward(t["q"], t["v"], t["decay"], t["dy"], t["rho_init"], t["rho_norm_init"], f[3],
                           d_rho_final=t["d_rho_final"], d_rho_norm_final=t["d_rho_norm_final"])
        torch.cuda.synchronize()
        out[variant] = dict(zip(("y", "rho_final", "rho_norm_final", "ckpt"), f), **g)
    b = out["sequential"]
    for variant in ("chunked", "split_backward"):
        a = out[variant]
        for k in a:
            ref = b[k].cpu().numpy().astype(np.float64)
            scale = float(np.abs(ref).mean()) if k == "ddecay" else 0.0
            _close(f"{k} {variant} vs sequential", a[k].cpu().numpy(), ref, scale)
