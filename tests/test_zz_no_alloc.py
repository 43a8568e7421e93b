"""The backward entry point that allocates no device memory.

Some callers of this library cannot allocate device memory: code recording a
CUDA graph that must not contain allocation nodes, or a framework that owns
every device byte through its own allocator. wkv7_backward_noalloc serves
them: its own checkpointing forward writes into a fixed scratch array of the
library instead of a cudaMallocAsync workspace. This file checks it, through
the C ABI, against the allocating wkv7_backward on the same inputs, on two
calls in a row (the scratch keeps whatever the previous call left in it), and
that a problem larger than the scratch is refused. Collected last on purpose.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")
TOL = 1e-4  # the fp32 parity bar used by every GPU test: |x - ref| <= TOL * (1 + |ref|)


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__  # noqa: F401
    from linear_rnn_state_gb300 import _build, inputs, wkv7

    _build.build()
    wkv7.load()
    torch.cuda.set_device(0)
    return inputs, wkv7


def _case(inputs, seed, B=2, T=300, H=4, N=64):
    dev = torch.device("cuda:0")
    d = inputs.generate(B, T, H, N, "f32", 0.1, seed=seed)
    t = {n: torch.from_numpy(d[n]).to(dev) for n in NAMES + ("dy",)}
    t["s_init"] = torch.from_numpy(d["s_init"].astype(np.float32)).to(dev)
    return t


def _close(got, ref):
    got = got.double()
    ref = ref.double()
    return bool(((got - ref).abs() <= TOL * (1.0 + ref.abs())).all())


def test_noalloc_backward_matches_the_allocating_backward_twice(env):
    inputs, wkv7 = env
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((21, 22)):
        t = _case(inputs, seed)
        B, T, H, N = t["r"].shape
        ref = wkv7.backward(*(t[n] for n in NAMES), t["dy"], t["s_init"], None, 0)
        out = {n: torch.full((B, T, H, N), float("nan"), device=t["r"].device) for n in GRADS}
        out["dS_init"] = torch.full((B, H, N, N), float("nan"), device=t["r"].device)
        rc = wkv7.wkv7_backward_noalloc(*(t[n].data_ptr() for n in NAMES), t["dy"].data_ptr(),
                                        t["s_init"].data_ptr(), *(out[n].data_ptr() for n in GRADS),
                                        out["dS_init"].data_ptr(), B, T, H, N, stream)
        assert rc == wkv7.OK, wkv7.last_error()
        wkv7.status()
        for n in GRADS + ("dS_init",):
            assert _close(out[n], ref[n]), f"call {call}: {n} differs from wkv7_backward"


def test_noalloc_refuses_problems_beyond_its_scratch(env):
    _, wkv7 = env
    fake = [0x7F0000000000 + i * (1 << 36) for i in range(15)]  # aligned, never dereferenced
    rc = wkv7.wkv7_backward_noalloc(*fake, 1, 65536, 40, 64, None)
    assert rc == wkv7.ERR_INVALID
    assert "fixed scratch" in wkv7.last_error()
