"""GPU parity of the split backward's tcgen05 output kernel.

The split backward (wkv7_backward_bf16 at N = 64 with 16-step checkpoints)
forms every chunk's gradients in a per-chunk output pass. The product library
runs it on warp-level mma.sync products; the same pass also exists with its
products on the 5th-generation tensor cores (tcgen05.mma, accumulators in
tensor memory, operands fed by TMA and shared-memory descriptors), selectable
in the debug build (include/wkv7_debug.h, wkv7_debug_out_kernel). This file
holds that kernel to the fp64 oracle with the bf16 bar of parity_bars on the
cases that exercise it: ragged tails, a carried state and a final-state
gradient, chunks run step by step, decays given as logits, and more tasks
than the persistent grid has CTAs; and to the default kernel's results.
"""
import ctypes

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
    torch.cuda.set_device(0)
    dbg = wkv7.load(_build.DEBUG_LIB)
    dbg.wkv7_debug_out_kernel.argtypes = [ctypes.c_int]
    yield oracle, inputs, dbg
    dbg.wkv7_debug_out_kernel(0)


def _bf16_bits(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _run(dbg, d, names, B, T, H, s0, dsf, logit, which):
    dev = torch.device("cuda:0")
    sp = torch.cuda.current_stream().cuda_stream
    t = {n: torch.from_numpy(d[n]).view(torch.bfloat16).to(dev) for n in names + ("dy",)}
    ck = torch.empty((B, H, (T + 15) // 16, 64, 64), device=dev)
    y = torch.empty((B, T, H, 64), dtype=torch.bfloat16, device=dev)
    fwd = dbg.wkv7_forward_logit_bf16 if logit else dbg.wkv7_forward_bf16
    assert fwd(*(t[n].data_ptr() for n in names), None if s0 is None else s0.data_ptr(), y.data_ptr(), None,
               ck.data_ptr(), 16, B, T, H, 64, sp) == 0
    g = {n: torch.full((B, T, H, 64), float("nan"), device=dev) for n in GRADS}
    dS = torch.full((B, H, 64, 64), float("nan"), device=dev)
    dbg.wkv7_debug_out_kernel(which)
    bwd = dbg.wkv7_backward_logit_bf16 if logit else dbg.wkv7_backward_segment_bf16
    rc = bwd(*(t[n].data_ptr() for n in names), t["dy"].data_ptr(), None if s0 is None else s0.data_ptr(),
             None if dsf is None else dsf.data_ptr(), ck.data_ptr(), 16, *(g[n].data_ptr() for n in GRADS),
             dS.data_ptr(), B, T, H, 64, sp)
    dbg.wkv7_debug_out_kernel(0)
    assert rc == 0, dbg.wkv7_last_error().decode()
    assert dbg.wkv7_status(sp) == 0
    g["dS_init"] = dS
    return {n: x.cpu().numpy() for n, x in g.items()}


@pytest.mark.parametrize("case", ["ragged", "state_and_final_gradient", "step_by_step_chunks", "logits",
                                  "more_tasks_than_ctas"])
def test_tc_output_kernel_parity(env, case):
    oracle, inputs, dbg = env
    B, T, H = {"more_tasks_than_ctas": (4, 1040, 32)}.get(case, (2, 130, 3))
    state = case == "state_and_final_gradient"
    d = dict(inputs.generate(B, T, H, 64, "bf16", 0.1 if state else None, seed=90 + len(case)))
    logit = case == "logits"
    names = ("r", "z", "k", "v", "a", "b") if logit else NAMES
    if logit:
        d["z"] = inputs.generate_logits(B, T, H, 64, "bf16", seed=91)
    if case == "step_by_step_chunks":
        w = inputs.as_f64(d["w"], "bf16").copy()
        w[0, 32:48, 0, :] = 0.0
        w[1, 70, 2, 5] = 20.0
        d["w"] = _bf16_bits(w)
    dev = torch.device("cuda:0")
    s0_np = d["s_init"].astype(np.float32) if state else None
    s0 = None if s0_np is None else torch.from_numpy(s0_np).to(dev)
    dsf_np = np.random.default_rng(5).standard_normal((B, H, 64, 64)).astype(np.float32) if state else None
    dsf = None if dsf_np is None else torch.from_numpy(dsf_np).to(dev)
    got = _run(dbg, d, names, B, T, H, s0, dsf, logit, 1)
    ref_kernel = _run(dbg, d, names, B, T, H, s0, dsf, logit, 0)
    o = {n: inputs.as_f64(d[n], "bf16") for n in names + ("dy",)}
    s064 = None if s0_np is None else s0_np.astype(np.float64)
    dsf64 = None if dsf_np is None else dsf_np.astype(np.float64)
    if logit:
        g_ref = oracle.backward_logit(*(o[n] for n in names), o["dy"], s064, dsf64)
    else:
        g_ref = oracle.backward(*(o[n] for n in names), o["dy"], s064, dsf64)
    gname = "dz" if logit else "dw"
    for n in ("dr", "dw", "dk", "dv", "da", "db"):
        ref = g_ref[gname if n == "dw" else n]
        check_bf16(f"{gname if n == 'dw' else n} ({case}, tcgen05)", got[n], ref)
        check_bf16(f"{gname if n == 'dw' else n} ({case}, tcgen05 vs mma.sync)", got[n], ref_kernel[n])
    check_bf16(f"dS_init ({case}, tcgen05)", got["dS_init"], g_ref["dS_init"], "state")
