"""GPU parity of the scan with the decay given as logits (wkv7_forward_logit_bf16,
wkv7_backward_logit_bf16: w = exp(-0.606531 sigmoid(z)) formed inside the
chunked kernels, dz returned in the place of dw) against the fp64 oracle's
forward_logit / backward_logit on the same bf16 inputs.

Bar as for every bf16 case (parity_bars.check_bf16): relative L2 <= 2e-2 per
output tensor and per (b, h, 16-step chunk), plus an element-wise guard.
"""
import numpy as np
import pytest

from parity_bars import check_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = ("r", "z", "k", "v", "a", "b")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__  # noqa: F401
    import oracle
    from linear_rnn_state_gb300 import _build, inputs, wkv7

    _build.build()
    wkv7.load()
    torch.cuda.set_device(0)
    return oracle, inputs, wkv7


def _rel(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    kind = "state" if name.startswith(("s_final", "dS_init")) else "seq"
    check_bf16(name, got, ref, kind)


def _data(inputs, B, T, H, seed, state):
    d = dict(inputs.generate(B, T, H, 64, "bf16", 0.1 if state else None, seed=seed))
    d["z"] = inputs.generate_logits(B, T, H, 64, "bf16", seed=seed)
    return d


def _dev(x):
    return torch.from_numpy(x).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("T", [16, 45, 130])
@pytest.mark.parametrize("state", [False, True])
def test_logit_parity(env, T, state):
    oracle, inputs, wkv7 = env
    B, H = 2, 3
    d = _data(inputs, B, T, H, seed=50 + T, state=state)
    t = {n: _dev(d[n]) for n in NAMES + ("dy",)}
    s0 = torch.from_numpy(d["s_init"].astype(np.float32)).cuda() if state else None
    dsf = (torch.from_numpy(np.random.default_rng(T).standard_normal((B, H, 64, 64)).astype(np.float32)).cuda()
           if state else None)
    y, sf, ck, _ = wkv7.forward_logit(*(t[n] for n in NAMES), s0)
    g = wkv7.backward_logit(*(t[n] for n in NAMES), t["dy"], s0, ck, dS_final=dsf)
    g2 = wkv7.backward_logit(*(t[n] for n in NAMES), t["dy"], s0, None, dS_final=dsf)  # own checkpoints
    wkv7.status()
    o = {n: inputs.as_f64(d[n], "bf16") for n in NAMES + ("dy",)}
    s064 = d["s_init"].astype(np.float32).astype(np.float64) if state else None
    dsf64 = dsf.cpu().numpy().astype(np.float64) if state else None
    y_ref, sf_ref = oracle.forward_logit(*(o[n] for n in NAMES), s064)
    g_ref = oracle.backward_logit(*(o[n] for n in NAMES), o["dy"], s064, dsf64)
    tag = f"T={T} state={state}"
    _rel(f"y {tag}", inputs.as_f64(y.view(torch.int16).cpu().numpy().view(np.uint16), "bf16"), y_ref)
    _rel(f"s_final {tag}", sf.cpu().numpy(), sf_ref)
    for n in ("dr", "dz", "dk", "dv", "da", "db", "dS_init"):
        _rel(f"{n} {tag}", g[n].cpu().numpy(), g_ref[n])
        assert torch.equal(g[n], g2[n]), f"{n}: own checkpoints differ"


def test_logit_extreme_logits(env):
    """Logits far in both tails: w -> 1 and w -> exp(-0.606531), sigmoid
    saturating in fp32."""
    oracle, inputs, wkv7 = env
    B, T, H = 1, 48, 2
    d = _data(inputs, B, T, H, seed=61, state=False)
    z = inputs.as_f64(d["z"], "bf16") * 30.0
    u = z.astype(np.float32).view(np.uint32).astype(np.uint64)
    d["z"] = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    t = {n: _dev(d[n]) for n in NAMES + ("dy",)}
    y, sf, ck, _ = wkv7.forward_logit(*(t[n] for n in NAMES))
    g = wkv7.backward_logit(*(t[n] for n in NAMES), t["dy"], None, ck)
    wkv7.status()
    o = {n: inputs.as_f64(d[n], "bf16") for n in NAMES + ("dy",)}
    g_ref = oracle.backward_logit(*(o[n] for n in NAMES), o["dy"])
    for n in ("dr", "dz", "dk", "dv", "da", "db"):
        _rel(n, g[n].cpu().numpy(), g_ref[n])


def test_logit_full_size_sampled(env):
    """B=4, T=4096, H=32, N=64 with logits, in the benchmark's launch
    configuration; the oracle recomputes every output of two (b, h) heads."""
    oracle, inputs, wkv7 = env
    B, T, H = 4, 4096, 32
    d = _data(inputs, B, T, H, seed=0, state=False)
    t = {n: _dev(d[n]) for n in NAMES + ("dy",)}
    y, sf, ck, _ = wkv7.forward_logit(*(t[n] for n in NAMES))
    g = wkv7.backward_logit(*(t[n] for n in NAMES), t["dy"], None, ck)
    wkv7.status()
    for bi, hi in ((0, 0), (3, 31)):
        o = {n: inputs.as_f64(d[n][bi:bi + 1, :, hi:hi + 1], "bf16") for n in NAMES + ("dy",)}
        y_ref, sf_ref = oracle.forward_logit(*(o[n] for n in NAMES))
        g_ref = oracle.backward_logit(*(o[n] for n in NAMES), o["dy"])
        yg = y[bi:bi + 1, :, hi:hi + 1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        _rel(f"y ({bi},{hi})", inputs.as_f64(yg, "bf16"), y_ref)
        _rel(f"s_final ({bi},{hi})", sf[bi:bi + 1, hi:hi + 1].cpu().numpy(), sf_ref)
        for n in ("dr", "dz", "dk", "dv", "da", "db"):
            _rel(f"{n} ({bi},{hi})", g[n][bi:bi + 1, :, hi:hi + 1].cpu().numpy(), g_ref[n])
