"""GPU parity of the chunked tensor-core kernels (bf16 inputs, N = 64,
checkpoints every multiple of 16 steps) against the fp64 oracle, for both
backward forms: the split one (wkv7_backward_bf16) and the fused one
(wkv7_backward_fused_bf16).

Bar (parity_bars.check_bf16): relative L2 <= 2e-2 over each output tensor and
over each of its (b, h, 16-step chunk) blocks, plus an element-wise guard;
the oracle reads exactly the bf16 values stored on the GPU. Cases span
several 16-step chunks, ragged tails, a carried initial state, and chunks
whose decays leave the range of the scaled form (w = 0, w > 16), which the
kernels run in the direct form.
"""
import numpy as np
import pytest

from parity_bars import check_bf16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")


@pytest.fixture(scope="module", params=["fused", "split"])
def env(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__  # noqa: F401
    import oracle
    from linear_rnn_state_gb300 import _build, inputs, wkv7

    _build.build()
    wkv7.load()
    torch.cuda.set_device(0)
    return oracle, inputs, wkv7, request.param == "fused"


def _bf16_bits(x):
    """float64 -> bf16 bit patterns, round to nearest even."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _check(env, d, C, s_init_std=None, use_ckpt=True, label=""):
    oracle, inputs, wkv7, fused = env
    dev = torch.device("cuda:0")
    t = {n: torch.from_numpy(d[n]).view(torch.bfloat16).to(dev) for n in NAMES + ("dy",)}
    s0_np = None if d.get("s_init") is None else d["s_init"].astype(np.float32)
    s0 = None if s0_np is None else torch.from_numpy(s0_np).to(dev)
    y, s_final, ckpt, C = wkv7.forward(*(t[n] for n in NAMES), s0, ckpt_every=C, want_ckpt=use_ckpt)
    # the fused form exists for 16-step checkpoints; longer intervals run the scalar kernels
    g = wkv7.backward(*(t[n] for n in NAMES), t["dy"], s0, ckpt if use_ckpt else None, C if use_ckpt else 0,
                      fused=fused and (C == 16 or not use_ckpt))
    wkv7.status()
    o = {n: inputs.as_f64(d[n], "bf16") for n in NAMES + ("dy",)}
    s0_64 = None if s0_np is None else s0_np.astype(np.float64)
    y_ref, sf_ref = oracle.forward(*(o[n] for n in NAMES), s0_64)
    g_ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s0_64)
    check_bf16(f"y{label}", y.float().cpu().numpy(), y_ref)
    check_bf16(f"s_final{label}", s_final.cpu().numpy(), sf_ref, "state")
    for n in GRADS:
        check_bf16(f"{n}{label}", g[n].cpu().numpy(), g_ref[n])
    check_bf16(f"dS_init{label}", g["dS_init"].cpu().numpy(), g_ref["dS_init"], "state")
    return y, s_final, ckpt


@pytest.mark.parametrize("T", [1, 15, 16, 17, 130, 300])
def test_chunked_ragged_lengths(env, T):
    inputs = env[1]
    d = inputs.generate(2, T, 3, 64, "bf16", None, seed=11)
    _check(env, d, 16, label=f" (T={T})")


@pytest.mark.parametrize("C,use_ckpt", [(16, True), (32, True), (48, True), (16, False)])
def test_chunked_checkpoint_intervals_and_carried_state(env, C, use_ckpt):
    inputs = env[1]
    d = inputs.generate(2, 200, 2, 64, "bf16", 0.1, seed=12)
    _check(env, d, C, use_ckpt=use_ckpt, label=f" (C={C}, ckpt={use_ckpt})")


def test_chunked_direct_form_chunks(env):
    """Chunks with w = 0 or w > 16 in some columns run step by step; the
    chunks around them stay on the scaled form."""
    inputs = env[1]
    d = dict(inputs.generate(1, 100, 2, 64, "bf16", 0.1, seed=13))
    w = inputs.as_f64(d["w"], "bf16").copy()
    w[0, 32:48, 0, :] = 0.0  # head 0: a whole chunk that forgets
    w[0, 70, 1, 5] = 20.0  # head 1: one growing column in chunk 4
    w[0, 99, 0, 63] = 0.0  # head 0: last (partial) chunk
    d["w"] = _bf16_bits(w)
    _check(env, d, 16, label=" (direct chunks)")


def test_chunked_outputs_overwritten(env):
    """Poisoned (NaN) outputs: every element is written."""
    _, inputs, wkv7, fused = env
    dev = torch.device("cuda:0")
    B, T, H, N, C = 1, 45, 3, 64, 16
    d = inputs.generate(B, T, H, N, "bf16", None, seed=14)
    t = {n: torch.from_numpy(d[n]).view(torch.bfloat16).to(dev) for n in NAMES + ("dy",)}
    stream = torch.cuda.current_stream().cuda_stream
    y = torch.full((B, T, H, N), float("nan"), dtype=torch.bfloat16, device=dev)
    sf = torch.full((B, H, N, N), float("nan"), device=dev)
    ck = torch.full((B, H, (T + C - 1) // C, N, N), float("nan"), device=dev)
    assert wkv7.wkv7_forward_bf16(*(t[n].data_ptr() for n in NAMES), None, y.data_ptr(), sf.data_ptr(),
                                  ck.data_ptr(), C, B, T, H, N, stream) == 0
    g = {n: torch.full((B, T, H, N), float("nan"), device=dev) for n in GRADS}
    dS = torch.full((B, H, N, N), float("nan"), device=dev)
    bwd = wkv7.wkv7_backward_fused_bf16 if fused else wkv7.wkv7_backward_segment_bf16
    assert bwd(*(t[n].data_ptr() for n in NAMES), t["dy"].data_ptr(), None, None, ck.data_ptr(), C,
               *(g[n].data_ptr() for n in GRADS), dS.data_ptr(), B, T, H, N, stream) == 0
    wkv7.status()
    for x in [y, sf, ck, dS] + list(g.values()):
        assert torch.isfinite(x).all()


def test_chunked_checkpoints_are_states(env):
    """Checkpoint c is the state before step 16c: a forward over the first 16c
    steps ends in exactly that state (same chunks, same arithmetic)."""
    _, inputs, wkv7, fused = env
    dev = torch.device("cuda:0")
    B, T, H, N, C = 1, 70, 2, 64, 16
    d = inputs.generate(B, T, H, N, "bf16", 0.1, seed=15)
    t = {n: torch.from_numpy(d[n]).view(torch.bfloat16).to(dev) for n in NAMES}
    s0 = torch.from_numpy(d["s_init"].astype(np.float32)).to(dev)
    _, _, ck, _ = wkv7.forward(*(t[n] for n in NAMES), s0, ckpt_every=C)
    torch.testing.assert_close(ck[:, :, 0], s0, rtol=0, atol=0)
    for c in range(1, T // C + 1):
        _, sf, _, _ = wkv7.forward(*(t[n][:, : c * C].contiguous() for n in NAMES), s0, ckpt_every=C)
        torch.testing.assert_close(ck[:, :, c], sf, rtol=0, atol=0)
