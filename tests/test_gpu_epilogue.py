"""GPU parity of the forward with the time-mix epilogue fused
(wkv7_forward_epilogue_bf16: group norm per head + bonus, "rx_pretrain.c")
against the fp64 oracles: the scan's (oracle) followed by the epilogue's
(oracle/epilogue_oracle.py), on the same bf16 inputs; the decay given as w
and as logits.

Bars: out, nv (the normalized y), the per-row stats (rstd, bonus) and every
gradient held to the bf16 bar of parity_bars.check_bf16 (relative L2 2e-2 per
tensor and per (b, h, 16-step chunk), plus an element-wise guard); the state
outputs (s_final, checkpoints) bit-equal to the plain forward's, which the
epilogue does not touch.
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


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__  # noqa: F401
    import oracle
    from linear_rnn_state_gb300 import _build, inputs, wkv7

    _build.build()
    wkv7.load()
    spec = importlib.util.spec_from_file_location("epilogue_oracle", os.path.join(ROOT, "oracle", "epilogue_oracle.py"))
    epi = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(epi)
    torch.cuda.set_device(0)
    return oracle, epi, inputs, wkv7


def _rel(name, got, ref):
    """The bf16 bar of parity_bars.check_bf16; states and [H][N] parameter
    gradients are one block each, per-step outputs are checked per chunk."""
    got = np.asarray(got, dtype=np.float64)
    kind = "state" if name.startswith(("dS_init", "dln_w", "dln_b", "dr_k")) else "seq"
    check_bf16(name, got, ref, kind)


def _bf(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _params(H, seed):
    rng = np.random.default_rng(seed)
    return (rng.uniform(0.5, 1.5, (H, 64)).astype(np.float32), (0.1 * rng.standard_normal((H, 64))).astype(np.float32),
            (0.5 * rng.standard_normal((H, 64))).astype(np.float32))


def _run(env, B, T, H, seed, logit, state, check_heads=None):
    oracle, epi, inputs, wkv7 = env
    d = dict(inputs.generate(B, T, H, 64, "bf16", 0.1 if state else None, seed=seed))
    if logit:
        d["w"] = inputs.generate_logits(B, T, H, 64, "bf16", seed=seed)
    t = {n: torch.from_numpy(d[n]).view(torch.bfloat16).cuda() for n in NAMES}
    s0 = torch.from_numpy(d["s_init"].astype(np.float32)).cuda() if state else None
    ln_w, ln_b, r_k = _params(H, seed)
    pt = [torch.from_numpy(x).cuda() for x in (ln_w, ln_b, r_k)]
    out, nv, stats, sf, ck = wkv7.forward_epilogue(*(t[n] for n in NAMES), *pt, s0, decay_is_logit=logit)
    fwd = wkv7.forward_logit if logit else wkv7.forward
    if logit:
        _, sf2, ck2, _ = fwd(*(t[n] for n in NAMES), s0)
    else:
        _, sf2, ck2, _ = fwd(*(t[n] for n in NAMES), s0, ckpt_every=16)
    wkv7.status()
    assert torch.equal(sf, sf2) and torch.equal(ck, ck2), "the epilogue changed the state outputs"
    heads = check_heads or [(bi, hi) for bi in range(B) for hi in range(H)]
    for bi, hi in heads:
        o = {n: inputs.as_f64(d[n][bi:bi + 1, :, hi:hi + 1], "bf16") for n in NAMES}
        s064 = d["s_init"][bi:bi + 1, hi:hi + 1].astype(np.float32).astype(np.float64) if state else None
        y_ref, _ = (oracle.forward_logit if logit else oracle.forward)(*(o[n] for n in NAMES), s064)
        out_ref, st = epi.forward(y_ref, o["r"], o["k"], o["v"], ln_w[hi:hi + 1], ln_b[hi:hi + 1], r_k[hi:hi + 1])
        nv_ref = (y_ref - st["mean"][..., None]) * st["rstd"][..., None]
        tag = f"T={T} logit={logit} head=({bi},{hi})"
        sl = (slice(bi, bi + 1), slice(None), slice(hi, hi + 1))
        _rel(f"out {tag}", inputs.as_f64(_bf(out[sl]), "bf16"), out_ref)
        _rel(f"nv {tag}", inputs.as_f64(_bf(nv[sl]), "bf16"), nv_ref)
        g = stats[sl].cpu().numpy().astype(np.float64)
        _rel(f"rstd {tag}", g[..., 0], st["rstd"])
        _rel(f"bonus {tag}", g[..., 1], st["bonus"])


@pytest.mark.parametrize("T", [16, 45, 130])
@pytest.mark.parametrize("logit", [False, True])
def test_epilogue_parity(env, T, logit):
    _run(env, 2, T, 3, seed=80 + T, logit=logit, state=(T != 16))


def test_epilogue_full_size_sampled(env):
    _run(env, 4, 4096, 32, seed=0, logit=True, state=False, check_heads=[(0, 0), (3, 31)])


@pytest.mark.parametrize("T", [16, 45, 130])
@pytest.mark.parametrize("logit", [False, True])
def test_epilogue_backward_parity(env, T, logit):
    """wkv7_backward_epilogue_bf16 against the chained oracles: the epilogue's
    backward gives the scan's dy and the bonus and parameter gradients, the
    scan's backward the rest; dr, dk, dv are the sums of both."""
    oracle, epi, inputs, wkv7 = env
    B, H = 2, 3
    d = dict(inputs.generate(B, T, H, 64, "bf16", 0.1, seed=120 + T))
    if logit:
        d["w"] = inputs.generate_logits(B, T, H, 64, "bf16", seed=120 + T)
    t = {n: torch.from_numpy(d[n]).view(torch.bfloat16).cuda() for n in NAMES + ("dy",)}
    s0 = torch.from_numpy(d["s_init"].astype(np.float32)).cuda()
    ln_w, ln_b, r_k = _params(H, 7 + T)
    pt = [torch.from_numpy(x).cuda() for x in (ln_w, ln_b, r_k)]
    out, nv, stats, sf, ck = wkv7.forward_epilogue(*(t[n] for n in NAMES), *pt, s0, decay_is_logit=logit)
    g = wkv7.backward_epilogue(*(t[n] for n in NAMES), t["dy"], nv, stats, pt[0], pt[2], s0, ck,
                               decay_is_logit=logit)
    wkv7.status()
    o = {n: inputs.as_f64(d[n], "bf16") for n in NAMES + ("dy",)}
    s064 = d["s_init"].astype(np.float32).astype(np.float64)
    y_ref, _ = (oracle.forward_logit if logit else oracle.forward)(*(o[n] for n in NAMES), s064)
    ge = epi.backward(o["dy"], y_ref, o["r"], o["k"], o["v"], ln_w, ln_b, r_k)
    gs = (oracle.backward_logit if logit else oracle.backward)(*(o[n] for n in NAMES), ge["dy"], s064)
    dwn = "dz" if logit else "dw"
    ref = {"dr": gs["dr"] + ge["dr"], "dk": gs["dk"] + ge["dk"], "dv": gs["dv"] + ge["dv"], dwn: gs[dwn],
           "da": gs["da"], "db": gs["db"], "dS_init": gs["dS_init"], "dln_w": ge["dln_w"], "dln_b": ge["dln_b"],
           "dr_k": ge["dr_k"]}
    for n, r in ref.items():
        _rel(f"{n} T={T} logit={logit}", g[n].cpu().numpy(), r)
