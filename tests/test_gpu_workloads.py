"""Parity at the full sizes of the three large workloads, in the launch
configuration the benchmark times.

The two 4096-step workloads are checked whole: the fp64 oracle recomputes
every output of every (b, h) head on the host cores (about a second), and
every element is held to the bar (fp32 inputs |gpu - ref| <= 1e-4 (1 + |ref|);
bf16 inputs parity_bars.check_bf16, per tensor, per (b, h, 16-step chunk) and
per element). For the 65536-step workload the oracle recomputes a sample of
heads in full, and the rest is checked through properties that hold at any
size: every output finite and the per-row identity dr_t . r_t = dy_t . y_t
(y is linear in r_t, which enters nowhere else).
"""
import numpy as np
import pytest

from parity_bars import check_bf16, record_f32

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")

NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__  # noqa: F401
    import oracle
    from linear_rnn_state_gb300 import _build, configs, inputs, wkv7

    _build.build()
    wkv7.load()
    torch.cuda.set_device(0)
    return oracle, inputs, wkv7, configs


def _check(name, got, ref, storage, kind="seq"):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), name
    if storage == "bf16":
        check_bf16(name, got, ref, kind)
    else:
        err = np.abs(got - ref) / (1.0 + np.abs(ref))
        i = np.unravel_index(np.argmax(err), err.shape)
        record_f32(name, err.max())
        assert err.max() <= 1e-4, f"{name}: max scaled error {err.max():.3e} at {i}"


@pytest.mark.parametrize("name", ["rwkv7-0.1b-layer-fp32", "rwkv7-1.5b-layer-bf16", "long-carry-fp32"])
def test_full_size_workload(env, name):
    oracle, inputs, wkv7, configs = env
    wl = configs.WORKLOADS[name]
    B, T, H, N, st = wl.B, wl.T, wl.H, wl.N, wl.storage
    dev = torch.device("cuda:0")
    d = inputs.generate(B, T, H, N, st, wl.s_init_std, seed=0)
    t = {}
    for n in NAMES + ("dy",):
        x = torch.from_numpy(d[n])
        t[n] = (x.view(torch.bfloat16) if st == "bf16" else x).to(dev)
    s0_np = None if d["s_init"] is None else d["s_init"].astype(np.float32)
    s0 = None if s0_np is None else torch.from_numpy(s0_np).to(dev)
    C = wl.ckpt_every if st == "f32" else wkv7.wkv7_default_ckpt_every(N, True)
    y, s_final, ckpt, C = wkv7.forward(*(t[n] for n in NAMES), s0, ckpt_every=C)
    g = wkv7.backward(*(t[n] for n in NAMES), t["dy"], s0, ckpt, C)
    wkv7.status()
    del ckpt

    # properties over every row of every head
    yf = y.float()
    lhs = (g["dr"] * t["r"].float()).sum(-1).double()
    rhs = (t["dy"].float() * yf).sum(-1).double()
    rel = (torch.linalg.vector_norm(lhs - rhs) / torch.linalg.vector_norm(rhs)).item()
    assert rel <= (2e-2 if st == "bf16" else 1e-4), f"dr.r vs dy.y: {rel:.3e}"
    for n in GRADS:
        assert torch.isfinite(g[n]).all(), n
    assert torch.isfinite(yf).all()

    o = {n: inputs.as_f64(d[n], st) for n in NAMES + ("dy",)}
    s064 = None if s0_np is None else s0_np.astype(np.float64)
    if T <= 4096:  # every head, every output, against the oracle
        y_ref, sf_ref = oracle.forward(*(o[n] for n in NAMES), s064)
        g_ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s064)
        _check("y", yf.cpu().numpy(), y_ref, st)
        _check("s_final", s_final.cpu().numpy(), sf_ref, st, "state")
        for n in GRADS:
            _check(n, g[n].cpu().numpy(), g_ref[n], st)
        _check("dS_init", g["dS_init"].cpu().numpy(), g_ref["dS_init"], st, "state")
        return

    # sampled heads in full against the oracle
    heads = [(0, 0), (B - 1, H - 1)]
    y_ref, sf_ref, g_ref = oracle.backward_heads(*(o[n] for n in NAMES), o["dy"], s064, heads)
    for p, (bi, hi) in enumerate(heads):
        _check(f"y[{bi},{hi}]", y[bi, :, hi].float().cpu().numpy(), y_ref[p], st)
        _check(f"s_final[{bi},{hi}]", s_final[bi, hi].cpu().numpy(), sf_ref[p], st, "state")
        for n in GRADS:
            _check(f"{n}[{bi},{hi}]", g[n][bi, :, hi].cpu().numpy(), g_ref[n][p], st)
        _check(f"dS_init[{bi},{hi}]", g["dS_init"][bi, hi].cpu().numpy(), g_ref["dS_init"][p], st, "state")
