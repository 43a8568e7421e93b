"""Host-side checks of the C ABI (no GPU needed): the library loads and exports
every function include/wkv7.h declares, and invalid arguments come back as
the documented status codes before anything touches a device."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wkv7.h")

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced by these calls
MB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
    from linear_rnn_state_gb300 import _build, wkv7

    _build.build()
    return wkv7


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wkv7_\w+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    declared = _declared_functions()
    assert declared, "no functions found in the header"
    raw = lib.load()
    for name in declared:
        assert hasattr(raw, name), f"{name} declared in wkv7.h but not exported"
    assert sorted(lib.EXPORTS) == declared


def test_debug_hook_only_in_the_debug_build(lib):
    """include/wkv7_debug.h's entry points are exported by libwkv7_debug.so
    alone; the product library does not carry them."""
    from linear_rnn_state_gb300 import _build

    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "wkv7_debug.h")).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(wkv7_\w+)\s*\(", text)))
    assert names == ["wkv7_debug_cut_extents", "wkv7_debug_out_kernel", "wkv7_debug_skip_last_load"]
    dbg = lib.load(_build.DEBUG_LIB)
    for n in names:
        assert hasattr(dbg, n)
        assert not hasattr(lib.load(), n)
    for n in lib.EXPORTS:  # the debug build is otherwise the same library
        assert hasattr(dbg, n)


def test_missing_library_fails_loudly(lib):
    with pytest.raises(RuntimeError, match="not built"):
        lib.load("/nonexistent/libwkv7.so")


def test_ckpt_bytes_and_default_interval(lib):
    assert lib.wkv7_ckpt_bytes(4, 4096, 32, 64, 16) == 4 * 32 * 256 * 64 * 64 * 4
    assert lib.wkv7_ckpt_bytes(1, 100, 1, 16, 7) == 15 * 16 * 16 * 4  # ceil(100/7) = 15
    assert lib.wkv7_ckpt_bytes(1, 10, 1, 48, 4) == 0
    assert lib.wkv7_ckpt_bytes(1, 10, 1, 16, 0) == 0
    for n in (16, 32, 64):
        assert lib.wkv7_default_ckpt_every(n, 0) >= 1
        assert lib.wkv7_default_ckpt_every(n, 1) >= 1
    assert lib.wkv7_default_ckpt_every(48, 0) == 0


def _fwd_args(B=1, T=8, H=1, N=16, **over):
    base = {n: FAKE + i * 64 * MB for i, n in enumerate(("r", "w", "k", "v", "a", "b", "s_init", "y", "s_final", "ckpt"))}
    base.update(over)
    return [base[n] for n in ("r", "w", "k", "v", "a", "b", "s_init", "y", "s_final", "ckpt")] + [
        over.get("C", 4), B, T, H, N, None]


def _bwd_args(B=1, T=8, H=1, N=16, **over):
    names = ("r", "w", "k", "v", "a", "b", "dy", "s_init", "ckpt", "dr", "dw", "dk", "dv", "da", "db", "dS_init")
    base = {n: FAKE + i * 64 * MB for i, n in enumerate(names)}
    base.update(over)
    p = [base[n] for n in names]
    return p[:9] + [over.get("C", 4)] + p[9:] + [B, T, H, N, None]


@pytest.mark.parametrize("fn", ["wkv7_forward", "wkv7_forward_bf16"])
@pytest.mark.parametrize("case,over", [
    ("bad_N", {"N": 48}),
    ("negative_T", {"T": -1}),
    ("null_input", {"k": None}),
    ("misaligned", {"v": FAKE + 4}),
    ("ckpt_every_zero", {"C": 0}),
    ("output_overlaps_input", {"y": FAKE + 64}),
    ("too_large", {"B": 1 << 14, "T": 1 << 16, "H": 64, "N": 64}),
])
def test_forward_rejects_invalid_arguments(lib, fn, case, over):
    over = dict(over)
    dims = {k: over.pop(k) for k in ("B", "T", "H", "N") if k in over}
    rc = getattr(lib, fn)(*_fwd_args(**dims, **over))
    assert rc == lib.ERR_INVALID, (case, rc, lib.last_error())
    assert lib.last_error()


@pytest.mark.parametrize("fn", ["wkv7_backward", "wkv7_backward_bf16"])
@pytest.mark.parametrize("case,over", [
    ("bad_N", {"N": 8}),
    ("null_dy", {"dy": None}),
    ("null_grad", {"da": None}),
    ("misaligned_grad", {"db": FAKE + 13 * 64 * MB + 8}),
    ("grad_overlaps_grad", {"dk": FAKE + 9 * 64 * MB + 32}),
    ("ckpt_every_negative_with_ckpt", {"C": -3}),
])
def test_backward_rejects_invalid_arguments(lib, fn, case, over):
    over = dict(over)
    dims = {k: over.pop(k) for k in ("B", "T", "H", "N") if k in over}
    rc = getattr(lib, fn)(*_bwd_args(**dims, **over))
    assert rc == lib.ERR_INVALID, (case, rc, lib.last_error())


def test_backward_workspace_allocation_failure_is_reported(lib, monkeypatch):
    monkeypatch.setenv("WKV7_FAIL_ALLOC", "1")
    rc = lib.wkv7_backward(*_bwd_args(ckpt=None, C=0))
    assert rc == lib.ERR_ALLOC
    assert "WKV7_FAIL_ALLOC" in lib.last_error()


def test_chunked_backward_reports_carry_workspace_failure(lib, monkeypatch):
    # bf16 inputs at N = 64 with 16-step checkpoints keep the carry of every chunk in a
    # workspace even when the checkpoints are given
    monkeypatch.setenv("WKV7_FAIL_ALLOC", "1")
    rc = lib.wkv7_backward_bf16(*_bwd_args(T=32, N=64, C=16))
    assert rc == lib.ERR_ALLOC
    assert "WKV7_FAIL_ALLOC" in lib.last_error()


def test_fused_backward_rejects_unsupported_shapes(lib):
    """The fused backward exists only in the chunked form: N = 64, 16-step
    checkpoints."""
    a = list(_bwd_args(T=32, N=32, C=16))
    a.insert(8, None)  # dS_final
    assert lib.wkv7_backward_fused_bf16(*a) == lib.ERR_INVALID
    assert "fused" in lib.last_error()
    a = list(_bwd_args(T=32, N=64, C=8))
    a.insert(8, None)
    assert lib.wkv7_backward_fused_bf16(*a) == lib.ERR_INVALID


def test_empty_problems_need_no_device(lib):
    # B*H == 0: nothing to do, every buffer may be NULL.
    assert lib.wkv7_forward(*([None] * 10), 4, 0, 8, 3, 16, None) == lib.OK
    assert lib.wkv7_backward(*([None] * 9), 4, *([None] * 7), 2, 8, 0, 16, None) == lib.OK
    # T == 0 without a final state / dS_init to write
    assert lib.wkv7_forward(*([None] * 10), 4, 2, 0, 3, 16, None) == lib.OK
    assert lib.wkv7_backward(*([None] * 9), 4, *([None] * 7), 2, 0, 3, 16, None) == lib.OK


def test_logit_entries_reject_unsupported_shapes(lib):
    """The decay-as-logits calls run only the N = 64, 16-step chunked kernels."""
    fwd = _fwd_args(N=32, C=16)
    assert lib.wkv7_forward_logit_bf16(*fwd) == lib.ERR_INVALID
    assert "logits" in lib.last_error()
    fwd = _fwd_args(N=64, C=8)
    assert lib.wkv7_forward_logit_bf16(*fwd) == lib.ERR_INVALID
    ptrs = [FAKE + i * 64 * MB for i in range(17)]
    bwd = ptrs[:10] + [8] + ptrs[10:17] + [1, 8, 1, 64, None]
    assert lib.wkv7_backward_logit_bf16(*bwd) == lib.ERR_INVALID
    bwd = ptrs[:10] + [16] + ptrs[10:17] + [1, 8, 1, 32, None]
    assert lib.wkv7_backward_logit_bf16(*bwd) == lib.ERR_INVALID


def test_epilogue_entry_rejects_unsupported_shapes_and_missing_parameters(lib):
    p = [FAKE + i * 64 * MB for i in range(15)]
    # r w k v a b s_init ln_w ln_b r_k out nv stats s_final ckpt, ckpt_every, logit, B, T, H, N, stream
    assert lib.wkv7_forward_epilogue_bf16(*p, 16, 0, 1, 8, 1, 32, None) == lib.ERR_INVALID
    assert lib.wkv7_forward_epilogue_bf16(*p, 8, 0, 1, 8, 1, 64, None) == lib.ERR_INVALID
    q = list(p)
    q[7] = None  # ln_w
    assert lib.wkv7_forward_epilogue_bf16(*q, 16, 0, 1, 8, 1, 64, None) == lib.ERR_INVALID
    q = list(p)
    q[11] = FAKE + 16  # nv overlapping r
    assert lib.wkv7_forward_epilogue_bf16(*q, 16, 0, 1, 8, 1, 64, None) == lib.ERR_INVALID


def test_epilogue_backward_entry_checks(lib, monkeypatch):
    p = [FAKE + i * 64 * MB for i in range(14)]
    g = [FAKE + (20 + i) * 64 * MB for i in range(10)]
    # N = 32 is not supported; a missing dln_w is refused; a failing workspace is reported
    assert lib.wkv7_backward_epilogue_bf16(*p, 16, 0, *g, 1, 8, 1, 32, None) == lib.ERR_INVALID
    q = list(g)
    q[7] = None
    assert lib.wkv7_backward_epilogue_bf16(*p, 16, 0, *q, 1, 8, 1, 64, None) == lib.ERR_INVALID
    monkeypatch.setenv("WKV7_FAIL_ALLOC", "1")
    assert lib.wkv7_backward_epilogue_bf16(*p, 16, 0, *g, 1, 8, 1, 64, None) == lib.ERR_ALLOC
