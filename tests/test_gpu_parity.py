"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Bar: fp32 inputs element by element, |gpu - ref| <= 1e-4 * (1 + |ref|);
bf16 inputs parity_bars.check_bf16: ||gpu - ref||_2 / ||ref||_2 <= 2e-2 over
each output tensor and each (b, h, 16-step chunk), plus an element-wise
guard. The oracle sees exactly the values stored in the GPU's input buffers
(bf16 or fp32, upcast to float64).
"""
import numpy as np
import pytest

from parity_bars import check_bf16, record_f32

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")
FP32_TOL = 1e-4


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


def _upload(d, storage, dev):
    out = {}
    for n in NAMES + ("dy",):
        x = torch.from_numpy(d[n])
        out[n] = (x.view(torch.bfloat16) if storage == "bf16" else x).to(dev)
    return out


def _s_init_f32(d):
    return None if d["s_init"] is None else d["s_init"].astype(np.float32)


def _oracle_inputs(inputs, d, storage):
    return {n: inputs.as_f64(d[n], storage) for n in NAMES + ("dy",)}


def _assert_close(name, got, ref, storage, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}{what}: non-finite values"
    if storage == "bf16":
        check_bf16(f"{name}{what}", got, ref, "state" if name in ("s_final", "dS_init") else "seq")
    else:
        err = np.abs(got - ref) / (1.0 + np.abs(ref))
        i = np.unravel_index(np.argmax(err), err.shape)
        record_f32(f"{name}{what}", err.max())
        assert err.max() <= FP32_TOL, f"{name}{what}: max scaled error {err.max():.3e} at {i}: {got[i]} vs {ref[i]}"


def _run_gpu(wkv7, t, s0, C, use_ckpt=True):
    y, s_final, ckpt, C = wkv7.forward(*(t[n] for n in NAMES), s0, ckpt_every=C, want_ckpt=use_ckpt)
    g = wkv7.backward(*(t[n] for n in NAMES), t["dy"], s0, ckpt if use_ckpt else None, C if use_ckpt else 0)
    wkv7.status()
    return y, s_final, g


def _full_parity(env, B, T, H, N, storage, s_init_std, C, seed=0, use_ckpt=True, zero_buffer=False, edit=None):
    oracle, inputs, wkv7 = env
    dev = torch.device("cuda:0")
    d = dict(inputs.generate(B, T, H, N, storage, s_init_std, seed=seed))
    if edit is not None:
        edit(d)
    t = _upload(d, storage, dev)
    s0_np = _s_init_f32(d)
    if s0_np is None and zero_buffer:
        s0_np = np.zeros((B, H, N, N), dtype=np.float32)
    s0 = None if s0_np is None else torch.from_numpy(s0_np).to(dev)
    y, s_final, g = _run_gpu(wkv7, t, s0, C, use_ckpt)
    o = _oracle_inputs(inputs, d, storage)
    s0_64 = None if s0_np is None else s0_np.astype(np.float64)
    y_ref, sf_ref = oracle.forward(*(o[n] for n in NAMES), s0_64)
    g_ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s0_64)
    _assert_close("y", y.float().cpu().numpy(), y_ref, storage)
    _assert_close("s_final", s_final.cpu().numpy(), sf_ref, storage)
    for n in GRADS + ("dS_init",):
        _assert_close(n, g[n].cpu().numpy(), g_ref[n], storage)


# ----------------------------------------------------- small, full compare --

@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_tiny_workload_every_checkpoint_interval(env, C):
    """B=1, T=64, H=2, N=16, fp32, zero initial state."""
    _full_parity(env, 1, 64, 2, 16, "f32", None, C)


def test_tiny_workload_internal_checkpoints(env):
    _full_parity(env, 1, 64, 2, 16, "f32", None, 16, use_ckpt=False)


def test_zero_state_buffer_equals_null(env):
    _full_parity(env, 1, 64, 2, 16, "f32", None, 16, zero_buffer=True)


def test_small_workload_with_carried_state(env):
    """B=2, T=512, H=4, N=64, fp32, s_init ~ N(0, 0.1); dS_init checked."""
    _full_parity(env, 2, 512, 4, 64, "f32", 0.1, 16)


@pytest.mark.parametrize("B,T,H,N,C", [
    (1, 1, 1, 64, 1),       # a single step
    (1, 3, 2, 64, 16),      # shorter than one staged block
    (2, 100, 3, 32, 7),     # ragged chunks (100 = 14*7 + 2)
    (1, 77, 2, 64, 20),     # chunk longer than the backward's shared-memory window
    (1, 50, 1, 16, 50),     # one chunk = the whole sequence
    (3, 37, 5, 16, 5),      # ragged, several heads
    (2, 20, 100, 16, 8),    # 200 heads: more CTAs than SMs
])
def test_edge_shapes(env, B, T, H, N, C):
    _full_parity(env, B, T, H, N, "f32", 0.3, C, seed=B * 1000 + T)


@pytest.mark.parametrize("N", [16, 32, 64])
def test_bf16_inputs(env, N):
    _full_parity(env, 2, 130, 3, N, "bf16", None, 8)


@pytest.mark.parametrize("C", [8, 16])
def test_decay_zero_and_one(env, C):
    """w = 0 (every step forgets) and w = 1 with a = b = 0 (pure accumulation);
    C = 16 runs the chunked kernels (w = 0 leaves the scaled form's range:
    every chunk step by step), C = 8 the scalar ones."""
    oracle, inputs, wkv7 = env
    dev = torch.device("cuda:0")
    B, T, H, N = 1, 33, 2, 64
    d = inputs.generate(B, T, H, N, "f32", 0.2, seed=5)
    for case in ("w0", "w1ab0"):
        e = dict(d)
        if case == "w0":
            e["w"] = np.zeros_like(d["w"])
        else:
            e["w"] = np.ones_like(d["w"])
            e["a"] = np.zeros_like(d["a"])
            e["b"] = np.zeros_like(d["b"])
        t = _upload(e, "f32", dev)
        s0_np = _s_init_f32(e)
        s0 = torch.from_numpy(s0_np).to(dev)
        y, s_final, g = _run_gpu(wkv7, t, s0, C)
        o = _oracle_inputs(inputs, e, "f32")
        y_ref, sf_ref = oracle.forward(*(o[n] for n in NAMES), s0_np.astype(np.float64))
        g_ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s0_np.astype(np.float64))
        _assert_close("y", y.cpu().numpy(), y_ref, "f32", f" ({case})")
        _assert_close("s_final", s_final.cpu().numpy(), sf_ref, "f32", f" ({case})")
        for n in GRADS + ("dS_init",):
            _assert_close(n, g[n].cpu().numpy(), g_ref[n], "f32", f" ({case})")


@pytest.mark.parametrize("B,T,H,C", [(1, 3, 2, 16), (1, 16, 1, 16), (2, 130, 3, 16), (1, 200, 2, 32)])
def test_fp32_chunked_shapes(env, B, T, H, C):
    """fp32 inputs at N = 64 with checkpoints on multiples of 16 steps: the
    chunked forward in split tf32; the chunked backward (carry chain + per-chunk
    output pass, split tf32) where the checkpoints come every 16 steps, the
    scalar backward at C = 32. Shorter than a chunk, exactly one chunk, ragged
    tails, carried state."""
    _full_parity(env, B, T, H, 64, "f32", 0.3, C, seed=7 * T + B)


def test_fp32_chunked_direct_form_chunks(env):
    """Chunks whose decays leave the scaled form's range run step by step in
    the chunked fp32 kernels: a whole chunk with w = 0 (head 0), one growing
    column (w = 20, head 1), a zero decay in the last, partial chunk."""
    def edit(d):
        w = d["w"].copy()
        w[0, 32:48, 0, :] = 0.0
        w[0, 70, 1, 5] = 20.0
        w[0, 99, 0, 63] = 0.0
        d["w"] = w

    _full_parity(env, 1, 100, 2, 64, "f32", 0.1, 16, seed=31, edit=edit)


def test_empty_sequence(env):
    _, _, wkv7 = env
    dev = torch.device("cuda:0")
    B, H, N = 2, 3, 16
    s0 = torch.randn(B, H, N, N, device=dev)
    s_final = torch.full_like(s0, float("nan"))
    dS = torch.full_like(s0, float("nan"))
    assert wkv7.wkv7_forward(*([None] * 6), s0.data_ptr(), None, s_final.data_ptr(), None, 4, B, 0, H, N,
                             torch.cuda.current_stream().cuda_stream) == 0
    assert wkv7.wkv7_backward(*([None] * 7), s0.data_ptr(), None, 4, *([None] * 6), dS.data_ptr(),
                              B, 0, H, N, torch.cuda.current_stream().cuda_stream) == 0
    wkv7.status()
    assert torch.equal(s_final, s0)
    assert torch.count_nonzero(dS) == 0


def test_outputs_are_overwritten_not_accumulated(env):
    """Poisoned (NaN) output buffers: every element must be written."""
    oracle, inputs, wkv7 = env
    dev = torch.device("cuda:0")
    B, T, H, N = 1, 45, 3, 32
    d = inputs.generate(B, T, H, N, "f32", 0.1, seed=9)
    t = _upload(d, "f32", dev)
    s0 = torch.from_numpy(_s_init_f32(d)).to(dev)
    C = 8
    stream = torch.cuda.current_stream().cuda_stream
    y = torch.full((B, T, H, N), float("nan"), device=dev)
    sf = torch.full((B, H, N, N), float("nan"), device=dev)
    ck = torch.full((B, H, (T + C - 1) // C, N, N), float("nan"), device=dev)
    assert wkv7.wkv7_forward(*(t[n].data_ptr() for n in NAMES), s0.data_ptr(), y.data_ptr(), sf.data_ptr(),
                             ck.data_ptr(), C, B, T, H, N, stream) == 0
    g = {n: torch.full((B, T, H, N), float("nan"), device=dev) for n in GRADS}
    dS = torch.full((B, H, N, N), float("nan"), device=dev)
    assert wkv7.wkv7_backward(*(t[n].data_ptr() for n in NAMES), t["dy"].data_ptr(), None, ck.data_ptr(), C,
                              *(g[n].data_ptr() for n in GRADS), dS.data_ptr(), B, T, H, N, stream) == 0
    wkv7.status()
    for x in [y, sf, ck, dS] + list(g.values()):
        assert torch.isfinite(x).all()


def test_checkpoints_are_states(env):
    """Checkpoint c holds the state before step c*C: the forward run for
    c*C steps ends in exactly that state."""
    _, inputs, wkv7 = env
    dev = torch.device("cuda:0")
    B, T, H, N, C = 1, 40, 2, 64, 8
    d = inputs.generate(B, T, H, N, "f32", 0.1, seed=3)
    t = _upload(d, "f32", dev)
    s0 = torch.from_numpy(_s_init_f32(d)).to(dev)
    _, _, ck, _ = wkv7.forward(*(t[n] for n in NAMES), s0, ckpt_every=C)
    torch.testing.assert_close(ck[:, :, 0], s0, rtol=0, atol=0)
    for c in range(1, T // C):
        _, sf, _, _ = wkv7.forward(*(t[n][:, : c * C].contiguous() for n in NAMES), s0, ckpt_every=C)
        torch.testing.assert_close(ck[:, :, c], sf, rtol=0, atol=0)
