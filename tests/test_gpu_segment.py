"""GPU parity of the segment backward (a gradient entering through the final
state) against the fp64 oracle, on every backward form: the scalar kernels
(fp32 and bf16 inputs, N = 16, 32, 64), the chunked tensor-core kernels (bf16
inputs at N = 64, split and fused) and their step-by-step chunks; and a
sequence cut into two segments against the whole sequence.

Bars as in test_gpu_parity.py: fp32 inputs |gpu - ref| <= 1e-4 (1 + |ref|)
element by element; bf16 inputs parity_bars.check_bf16 (relative L2 <= 2e-2
per tensor and per (b, h, 16-step chunk), plus an element-wise guard).
"""
import numpy as np
import pytest

from parity_bars import check_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")


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


def _close(name, got, ref, storage, kind="seq"):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), name
    if storage == "bf16":
        check_bf16(name, got, ref, kind)
    else:
        err = np.abs(got - ref) / (1.0 + np.abs(ref))
        assert err.max() <= 1e-4, f"{name}: max scaled error {err.max():.3e}"


def _bits_bf16(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _case(env, B, T, H, N, storage, C, seed, *, split=None, zero_chunk=False, use_ckpt=True):
    oracle, inputs, wkv7 = env
    dev = torch.device("cuda:0")
    d = dict(inputs.generate(B, T, H, N, storage, 0.2, seed=seed))
    if zero_chunk:  # a chunk that forgets: run step by step by every kernel
        w = inputs.as_f64(d["w"], storage).copy()
        w[0, 16:32, 0, :] = 0.0
        d["w"] = _bits_bf16(w) if storage == "bf16" else w.astype(np.float32)
    t = {}
    for n in NAMES + ("dy",):
        x = torch.from_numpy(d[n])
        t[n] = (x.view(torch.bfloat16) if storage == "bf16" else x).to(dev)
    s0_np = d["s_init"].astype(np.float32)
    dsf_np = np.random.default_rng(seed + 100).standard_normal((B, H, N, N)).astype(np.float32)
    s0, dsf = torch.from_numpy(s0_np).to(dev), torch.from_numpy(dsf_np).to(dev)
    _, _, ckpt, C = wkv7.forward(*(t[n] for n in NAMES), s0, ckpt_every=C, want_ckpt=use_ckpt)
    g = wkv7.backward(*(t[n] for n in NAMES), t["dy"], s0, ckpt if use_ckpt else None, C if use_ckpt else 0,
                      dS_final=dsf, fused=split is False)
    wkv7.status()
    o = {n: inputs.as_f64(d[n], storage) for n in NAMES + ("dy",)}
    g_ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s0_np.astype(np.float64), dsf_np.astype(np.float64))
    for n in GRADS:
        _close(f"{n} ({storage}, N={N}, T={T})", g[n].cpu().numpy(), g_ref[n], storage)
    _close(f"dS_init ({storage}, N={N}, T={T})", g["dS_init"].cpu().numpy(), g_ref["dS_init"], storage, "state")


@pytest.mark.parametrize("N", [16, 32, 64])
def test_segment_fp32_scalar_kernels(env, N):
    _case(env, 2, 45, 2, N, "f32", 16, seed=31)


def test_segment_fp32_internal_checkpoints(env):
    _case(env, 1, 70, 3, 32, "f32", 0, seed=32, use_ckpt=False)


def test_segment_bf16_scalar_kernels(env):
    _case(env, 2, 40, 2, 32, "bf16", 8, seed=33)


@pytest.mark.parametrize("split", [True, False])
@pytest.mark.parametrize("T", [16, 45, 130])
def test_segment_bf16_chunked(env, split, T):
    _case(env, 2, T, 3, 64, "bf16", 16, seed=34, split=split)


@pytest.mark.parametrize("split", [True, False])
def test_segment_bf16_chunked_step_by_step_chunk(env, split):
    _case(env, 1, 64, 2, 64, "bf16", 16, seed=35, split=split, zero_chunk=True)


def test_segment_fp32_step_by_step_chunk(env):
    _case(env, 1, 64, 2, 64, "f32", 16, seed=36, zero_chunk=True)


@pytest.mark.parametrize("storage", ["f32", "bf16"])
def test_two_segments_compose(env, storage):
    """Backward of [T1, T) with dS_final, then of [0, T1) with its dS_init,
    equals the backward of the whole sequence with dS_final."""
    oracle, inputs, wkv7 = env
    dev = torch.device("cuda:0")
    B, T, H, N, T1 = 2, 96, 2, 64, 48
    d = inputs.generate(B, T, H, N, storage, 0.2, seed=37)
    t = {}
    for n in NAMES + ("dy",):
        x = torch.from_numpy(d[n])
        t[n] = (x.view(torch.bfloat16) if storage == "bf16" else x).to(dev)
    s0 = torch.from_numpy(d["s_init"].astype(np.float32)).to(dev)
    dsf = torch.from_numpy(np.random.default_rng(37).standard_normal((B, H, N, N)).astype(np.float32)).to(dev)
    first = {n: t[n][:, :T1].contiguous() for n in t}
    second = {n: t[n][:, T1:].contiguous() for n in t}
    full = wkv7.backward(*(t[n] for n in NAMES), t["dy"], s0, dS_final=dsf)
    _, s_mid, _, _ = wkv7.forward(*(first[n] for n in NAMES), s0, ckpt_every=16)
    g2 = wkv7.backward(*(second[n] for n in NAMES), second["dy"], s_mid, dS_final=dsf)
    g1 = wkv7.backward(*(first[n] for n in NAMES), first["dy"], s0, dS_final=g2["dS_init"])
    wkv7.status()
    for n in GRADS:
        got = torch.cat([g1[n], g2[n]], dim=1).cpu().numpy()
        _close(f"{n} ({storage})", got, full[n].cpu().numpy().astype(np.float64), storage)
    _close(f"dS_init ({storage})", g1["dS_init"].cpu().numpy(), full["dS_init"].cpu().numpy().astype(np.float64),
           storage, "state")


def test_empty_segment_passes_the_gradient_through(env):
    _, _, wkv7 = env
    dev = torch.device("cuda:0")
    B, H, N = 2, 3, 64
    dsf = torch.randn((B, H, N, N), device=dev)
    dS = torch.full((B, H, N, N), float("nan"), device=dev)
    z = torch.empty((B, 0, H, N), dtype=torch.bfloat16, device=dev)
    g = {n: torch.empty((B, 0, H, N), device=dev) for n in GRADS}
    stream = torch.cuda.current_stream().cuda_stream
    rc = wkv7.wkv7_backward_segment_bf16(*([z.data_ptr()] * 7), None, dsf.data_ptr(), None, 16,
                                         *(g[n].data_ptr() for n in GRADS), dS.data_ptr(), B, 0, H, N, stream)
    assert rc == 0, wkv7.last_error()
    wkv7.status()
    assert torch.equal(dS, dsf)
