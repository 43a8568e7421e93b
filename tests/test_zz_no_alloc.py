"""The backward entry point that allocates no device memory.

Some callers of this library cannot allocate device memory: code recording a
CUDA graph that must not contain allocation nodes, or a framework that owns
every device byte through its own allocator. wkv7_backward_noalloc serves
them: its own checkpointing forward writes into a fixed scratch array of the
library instead of a cudaMallocAsync workspace.

This file checks it through the C ABI against the fp64 oracle, element by
element at the fp32 bar, and against the allocating wkv7_backward, on two
calls in a row of different shapes: the second call's checkpoints land on
scratch that the first call left holding other data, which the second must
overwrite before it reads. It records the call into a CUDA graph, checks that
the graph holds no allocation or free node, and replays it on new inputs
against the oracle. It also checks that a problem larger than the scratch is
refused. Collected last on purpose.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAMES = ("r", "w", "k", "v", "a", "b")
GRADS = ("dr", "dw", "dk", "dv", "da", "db")
TOL = 1e-4  # the fp32 parity bar of every GPU test: |x - ref| <= TOL * (1 + |ref|)


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


def _assert_close(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    i = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= TOL, f"{name}: max scaled error {err.max():.3e} at {i}: {got[i]} vs {ref[i]}"


@pytest.mark.parametrize("shapes", [((1, 97, 3, 64), (2, 300, 4, 64)), ((2, 300, 4, 64), (1, 40, 2, 32))])
def test_noalloc_backward_matches_the_oracle_on_two_calls(env, shapes):
    oracle, inputs, wkv7 = env
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    for call, (B, T, H, N) in enumerate(shapes):
        d = inputs.generate(B, T, H, N, "f32", 0.1, seed=21 + call)
        t = {n: torch.from_numpy(d[n]).to(dev) for n in NAMES + ("dy",)}
        s0_np = d["s_init"].astype(np.float32)
        s0 = torch.from_numpy(s0_np).to(dev)
        out = {n: torch.full((B, T, H, N), float("nan"), device=dev) for n in GRADS}
        out["dS_init"] = torch.full((B, H, N, N), float("nan"), device=dev)
        rc = wkv7.wkv7_backward_noalloc(*(t[n].data_ptr() for n in NAMES), t["dy"].data_ptr(), s0.data_ptr(),
                                        *(out[n].data_ptr() for n in GRADS), out["dS_init"].data_ptr(),
                                        B, T, H, N, stream)
        assert rc == wkv7.OK, wkv7.last_error()
        wkv7.status()
        o = {n: d[n].astype(np.float64) for n in NAMES + ("dy",)}
        ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s0_np.astype(np.float64))
        alloc = wkv7.backward(*(t[n] for n in NAMES), t["dy"], s0, None, 0)
        wkv7.status()
        for n in GRADS + ("dS_init",):
            got = out[n].cpu().numpy()
            _assert_close(f"call {call} {n} vs the oracle", got, ref[n])
            _assert_close(f"call {call} {n} vs wkv7_backward", got, alloc[n].cpu().numpy().astype(np.float64))


def test_noalloc_refuses_problems_beyond_its_scratch(env):
    wkv7 = env[2]
    fake = [0x7F0000000000 + i * (1 << 36) for i in range(15)]  # aligned, never dereferenced
    rc = wkv7.wkv7_backward_noalloc(*fake, 1, 65536, 40, 64, None)
    assert rc == wkv7.ERR_INVALID
    assert "fixed scratch" in wkv7.last_error()


def test_noalloc_backward_records_into_a_cuda_graph(env):
    """The call captured on a stream (thread-local capture mode, through the CUDA runtime
    this library shares with PyTorch): kernels and copies only, no allocation or free nodes;
    the instantiated graph replayed twice on new inputs written into the captured buffers."""
    import ctypes

    oracle, inputs, wkv7 = env
    rt = ctypes.CDLL("libcudart.so.13")
    vp = ctypes.c_void_p
    rt.cudaStreamBeginCapture.argtypes = [vp, ctypes.c_int]
    rt.cudaStreamEndCapture.argtypes = [vp, ctypes.POINTER(vp)]
    rt.cudaGraphGetNodes.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_size_t)]
    rt.cudaGraphNodeGetType.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    rt.cudaGraphInstantiate.argtypes = [ctypes.POINTER(vp), vp, ctypes.c_ulonglong]
    rt.cudaGraphLaunch.argtypes = [vp, vp]
    rt.cudaStreamSynchronize.argtypes = [vp]
    rt.cudaGraphExecDestroy.argtypes = [vp]
    rt.cudaGraphDestroy.argtypes = [vp]
    kKernel, kMemAlloc, kMemFree = 0, 10, 11  # cudaGraphNodeType values
    kThreadLocal = 1  # cudaStreamCaptureModeThreadLocal

    B, T, H, N = 1, 97, 3, 64
    dev = torch.device("cuda:0")
    d = inputs.generate(B, T, H, N, "f32", 0.1, seed=41)
    t = {n: torch.from_numpy(d[n]).to(dev) for n in NAMES + ("dy",)}
    s0 = torch.from_numpy(d["s_init"].astype(np.float32)).to(dev)
    out = {n: torch.empty((B, T, H, N), device=dev) for n in GRADS}
    out["dS_init"] = torch.empty((B, H, N, N), device=dev)
    args = ([t[n].data_ptr() for n in NAMES] + [t["dy"].data_ptr(), s0.data_ptr()] +
            [out[n].data_ptr() for n in GRADS] + [out["dS_init"].data_ptr()])
    side = torch.cuda.Stream(device=dev)
    st = vp(side.cuda_stream)
    torch.cuda.synchronize()
    # a first call outside the capture looks up the scratch and status addresses
    assert wkv7.wkv7_backward_noalloc(*args, B, T, H, N, side.cuda_stream) == wkv7.OK, wkv7.last_error()
    torch.cuda.synchronize()
    wkv7.status()

    graph, exe = vp(), vp()
    assert rt.cudaStreamBeginCapture(st, kThreadLocal) == 0
    rc = wkv7.wkv7_backward_noalloc(*args, B, T, H, N, side.cuda_stream)
    e = rt.cudaStreamEndCapture(st, ctypes.byref(graph))
    assert rc == wkv7.OK, wkv7.last_error()
    assert e == 0, f"cudaStreamEndCapture: {e}"
    try:
        count = ctypes.c_size_t(0)
        assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(count)) == 0
        nodes = (vp * count.value)()
        assert rt.cudaGraphGetNodes(graph, ctypes.cast(nodes, vp), ctypes.byref(count)) == 0
        types = []
        for i in range(count.value):
            ty = ctypes.c_int(-1)
            assert rt.cudaGraphNodeGetType(vp(nodes[i]), ctypes.byref(ty)) == 0
            types.append(ty.value)
        assert kMemAlloc not in types and kMemFree not in types, types
        assert types.count(kKernel) >= 2, types  # the checkpointing forward and the backward
        assert rt.cudaGraphInstantiate(ctypes.byref(exe), graph, 0) == 0
        for rep in range(2):
            d = inputs.generate(B, T, H, N, "f32", 0.1, seed=50 + rep)
            for n in NAMES + ("dy",):
                t[n].copy_(torch.from_numpy(d[n]))
            s0_np = d["s_init"].astype(np.float32)
            s0.copy_(torch.from_numpy(s0_np))
            for x in out.values():
                x.fill_(float("nan"))
            torch.cuda.synchronize()
            assert rt.cudaGraphLaunch(exe, st) == 0
            assert rt.cudaStreamSynchronize(st) == 0
            wkv7.status()
            o = {n: d[n].astype(np.float64) for n in NAMES + ("dy",)}
            ref = oracle.backward(*(o[n] for n in NAMES), o["dy"], s0_np.astype(np.float64))
            for n in GRADS + ("dS_init",):
                _assert_close(f"replay {rep} {n} vs the oracle", out[n].cpu().numpy(), ref[n])
    finally:
        if exe.value:
            rt.cudaGraphExecDestroy(exe)
        rt.cudaGraphDestroy(graph)
