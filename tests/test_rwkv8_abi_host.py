"""Host-side checks of the RWKV-8 C ABI (no GPU needed): the library exports
every function include/rwkv8.h declares, and invalid arguments, injected
workspace failures and empty problems come back as the documented status
codes before anything touches a device."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rwkv8.h")

FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced by these calls
MB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__  # noqa: F401
    from linear_rnn_state_gb300 import _build, rwkv8

    _build.build()
    return rwkv8


def test_exports_every_declared_function(lib):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    declared = sorted(set(re.findall(r"\b(rwkv8_\w+)\s*\(", text)))
    assert declared
    raw = lib.load()
    for name in declared:
        assert hasattr(raw, name), f"{name} declared in rwkv8.h but not exported"
    assert sorted(lib.EXPORTS) == declared


def test_ckpt_bytes(lib):
    assert lib.rwkv8_ckpt_bytes(4, 4096, 32, 64, 64) == 4 * 32 * 256 * (64 * 64 + 64) * 4
    assert lib.rwkv8_ckpt_bytes(1, 17, 1, 64, 64) == 2 * (64 * 64 + 64) * 4
    assert lib.rwkv8_ckpt_bytes(1, 16, 1, 32, 64) == 0
    assert lib.rwkv8_ckpt_bytes(-1, 16, 1, 64, 64) == 0


FWD_NAMES = ("q", "v", "decay", "rho_init", "rho_norm_init", "y", "rho_final", "rho_norm_final", "ckpt")
BWD_NAMES = ("q", "v", "decay", "dy", "rho_init", "rho_norm_init", "d_rho_final", "d_rho_norm_final", "ckpt", "dq",
             "dv", "ddecay", "d_rho_init", "d_rho_norm_init")


def _args(names, B=1, T=8, H=2, Hv=2, L=64, E=64, **over):
    base = {n: FAKE + i * 64 * MB for i, n in enumerate(names)}
    base.update(over)
    return [base[n] for n in names] + [B, T, H, Hv, L, E, None]


BAD = [
    ("q_null", {"q": None}),
    ("y_null", {"y": None}),
    ("misaligned_v", {"v": FAKE + 8}),
    ("L_not_64", {"L": 32}),
    ("E_not_64", {"E": 128}),
    ("value_heads", {"Hv": 3}),
    ("negative_T", {"T": -1}),
    ("y_overlaps_q", {"y": FAKE + 16}),
    ("too_many_heads", {"B": 1 << 14, "H": 1 << 14, "Hv": 1 << 14}),  # B * H must stay below 2^28
]


@pytest.mark.parametrize("case,over", BAD, ids=[c for c, _ in BAD])
def test_forward_rejects_invalid_arguments(lib, case, over):
    dims = {k: over.pop(k) for k in ("B", "T", "H", "Hv", "L", "E") if k in over}
    rc = lib.rwkv8_forward(*_args(FWD_NAMES, **dims, **over))
    assert rc == -2, (case, rc)
    assert lib.wkv7.last_error()


BAD_BWD = [
    ("dy_null", {"dy": None}),
    ("ddecay_null", {"ddecay": None}),
    ("dq_overlaps_dy", {"dq": FAKE + 3 * 64 * MB + 16}),
    ("dv_overlaps_dq", {"dv": FAKE + 9 * 64 * MB + 16}),
    ("misaligned_ckpt", {"ckpt": FAKE + 8 * 64 * MB + 4}),
    ("value_heads", {"Hv": 0}),
]


@pytest.mark.parametrize("case,over", BAD_BWD, ids=[c for c, _ in BAD_BWD])
def test_backward_rejects_invalid_arguments(lib, case, over):
    dims = {k: over.pop(k) for k in ("B", "T", "H", "Hv", "L", "E") if k in over}
    rc = lib.rwkv8_backward(*_args(BWD_NAMES, **dims, **over))
    assert rc == -2, (case, rc)


def test_backward_workspace_failure_is_reported(lib, monkeypatch):
    monkeypatch.setenv("WKV7_FAIL_ALLOC", "1")
    rc = lib.rwkv8_backward(*_args(BWD_NAMES))
    assert rc == -1
    assert "WKV7_FAIL_ALLOC" in lib.wkv7.last_error()


def test_forward_checkpoint_workspace_failure_is_reported(lib, monkeypatch):
    # without a checkpoint buffer the per-chunk readout needs a workspace for the chunk states
    monkeypatch.setenv("WKV7_FAIL_ALLOC", "1")
    monkeypatch.delenv("RWKV8_SEQUENTIAL", raising=False)
    rc = lib.rwkv8_forward(*_args(FWD_NAMES, ckpt=None))
    assert rc == -1
    assert "WKV7_FAIL_ALLOC" in lib.wkv7.last_error()


def test_empty_problems_need_no_device(lib):
    # B*H == 0: nothing to do, every buffer may be NULL
    assert lib.rwkv8_forward(*([None] * 9), 0, 8, 2, 2, 64, 64, None) == 0
    assert lib.rwkv8_backward(*([None] * 14), 2, 8, 0, 0, 64, 64, None) == 0
    # T == 0 with no state to pass on (decay stays required)
    assert lib.rwkv8_forward(None, None, FAKE, *([None] * 6), 2, 0, 2, 2, 64, 64, None) == 0
    assert lib.rwkv8_forward(*([None] * 9), 2, 0, 2, 2, 64, 64, None) == -2
