"""The C-ABI library: it builds, loads, exports every declared entry point, and
rejects bad arguments on the host before touching any device (CPU only)."""
import ctypes
import os
import re

import pytest

import attention_pipelining_gb300 as ap
from attention_pipelining_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ap.build()
    return ap._load()


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*((?:attn|chunk_scan)_[a-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_expected_entry_points():
    names = _declared_functions()
    assert set(ap.EXPORTS) <= set(names), names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_built_for_sm103a_only():
    assert _build.GENCODE == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in range(6):
        s = ap.status_string(code)
        assert isinstance(s, str) and s
    assert ap.status_string(99) == "unknown status"
    assert lib.attn_version() >= 100


# Fake, never-dereferenced device addresses: validation must reject or accept
# them without any CUDA call, so these run without a GPU.
A = 0x10000  # 16-byte aligned
GOOD = dict(B=1, H_q=4, H_kv=2, S_q=128, S_kv=128, D=128, causal=0, scale=0.125)


def _call(lib, q=A, k=A, v=A, o=A, lse=A, **kw):
    a = dict(GOOD)
    a.update(kw)
    return lib.attn_fwd(q, k, v, o, lse, a["B"], a["H_q"], a["H_kv"], a["S_q"], a["S_kv"], a["D"],
                        a["causal"], a["scale"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1), (dict(lse=None), 1),
    (dict(B=0), 1), (dict(H_q=0), 1), (dict(H_kv=0), 1), (dict(S_q=0), 1), (dict(S_kv=-3), 1),
    (dict(D=0), 1), (dict(H_q=3, H_kv=2), 1), (dict(causal=2), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(scale=float("-inf")), 1),
    (dict(D=96), 2), (dict(D=256), 2), (dict(D=32), 2), (dict(B=70000), 2),
    (dict(q=A + 8), 3), (dict(k=A + 2), 3), (dict(v=A + 4), 3), (dict(o=A + 1), 3), (dict(lse=A + 4), 3),
])
def test_validation_rejects_before_launch(lib, kw, code):
    assert _call(lib, **kw) == code


@pytest.mark.parametrize("scale", [-0.5, -0.0, 0.0, -1e30])
def test_validation_accepts_any_finite_scale(lib, scale):
    # the definition admits any real scale: a negative one passes the scale
    # check and the call stops at the next rule (a misaligned pointer here),
    # still before any CUDA call
    assert _call(lib, scale=scale, o=A + 8) == 3


def test_host_entry_rejects_null_host_buffers(lib):
    args = [A, A, A, A, A, A, A, A, A, A, 1, 4, 2, 128, 128, 128, 0, ctypes.c_float(0.1), None]
    for i in range(5):
        bad = list(args)
        bad[i] = None
        assert lib.attn_fwd_host(*bad) == 1


def test_bwd_host_entry_rejects_before_queuing(lib):
    """attn_bwd_host: a null host buffer, then the device-side rules of
    attn_bwd (fake, never-dereferenced device addresses), all on the host."""
    dims = [1, 4, 2, 128, 128, 128, 0, ctypes.c_float(0.1), None]
    ws_bytes = lib.attn_bwd_workspace_bytes(1, 4, 2, 128, 128)
    assert ws_bytes > 0

    def call(host=None, dev=None, ws=A, nbytes=ws_bytes, d=dims):
        host = host or [A] * 9
        dev = dev or [A] * 9
        return lib.attn_bwd_host(*host, *dev, ws, nbytes, *d)

    for i in range(9):
        host = [A] * 9
        host[i] = None
        assert call(host=host) == 1                   # null host buffer
    for i in range(9):
        dev = [A] * 9
        dev[i] = None
        assert call(dev=dev) == 1                     # null device buffer
    assert call(ws=None) == 1                         # no workspace
    assert call(nbytes=ws_bytes - 1) == 1             # too small a workspace
    assert call(ws=A + 16) == 3                       # workspace not 256-byte aligned
    dev = [A] * 9
    dev[5] = A + 8
    assert call(dev=dev) == 3                         # misaligned dout
    assert call(d=[1, 4, 2, 128, 128, 96, 0, ctypes.c_float(0.1), None]) == 2   # D = 96
    assert call(d=[1, 3, 2, 128, 128, 128, 0, ctypes.c_float(0.1), None]) == 1  # H_q % H_kv


def test_selftest_entry_validation(lib):
    assert lib.attn_selftest_qk(None, A, A, 128, None) == 1
    assert lib.attn_selftest_qk(A, A, A, 96, None) == 2
    assert lib.attn_selftest_pv(A, A + 4, A, 64, None) == 3


def test_trace_entry_validation(lib):
    base = [A, A, A, A, A, 1, 2, 2, 128, 128, 128, 0, ctypes.c_float(0.1)]
    assert lib.attn_fwd_trace(*base, None, 1, 1, None) == 1
    assert lib.attn_fwd_trace(*base, A, 0, 1, None) == 1
    assert lib.attn_fwd_trace(*base, A, 1, 0, None) == 1
    assert lib.attn_fwd_trace(*base, A + 4, 1, 1, None) == 3


def test_timeout_test_entry_validation(lib):
    base = [A, A, A, A, A, 1, 2, 2, 128, 128, 128, 0, ctypes.c_float(0.1)]
    assert lib.attn_fwd_timeout_test(*base, -1, 20_000_000, None) == 1     # no block to drop
    assert lib.attn_fwd_timeout_test(*base, 1, 10, None) == 1              # budget too short
    assert lib.attn_fwd_timeout_test(*base, 1, 10**10, None) == 1          # budget too long
    bad = [A, A, A, A, A, 1, 2, 2, 128, 128, 96, 0, ctypes.c_float(0.1)]
    assert lib.attn_fwd_timeout_test(*bad, 1, 20_000_000, None) == 2


def test_splitkv_entry_validation(lib):
    ws = A
    base = [A, A, A, A, A]
    dims = [1, 4, 2, 1, 4096, 128, 0, ctypes.c_float(0.1)]
    assert lib.attn_fwd_splitkv(*base, None, 1 << 20, *dims, 4, None) == 1        # no workspace
    assert lib.attn_fwd_splitkv(*base, ws + 16, 1 << 20, *dims, 4, None) == 3     # not 256-aligned
    assert lib.attn_fwd_splitkv(*base, ws, 1 << 20, *dims, 129, None) == 2        # too many splits
    assert lib.attn_splitkv_workspace_bytes(1, 4, 1, 128, 4) == 4 * 4 * (128 * 4) + 4 * 4 * 4 + (
        (256 - (4 * 4 * 128 * 4) % 256) % 256)
    assert lib.attn_splitkv_workspace_bytes(1, 4, 1, 96, 4) == 0
    assert lib.attn_splitkv_default_splits(1, 3, 2, 1, 100, 0) == 0


def test_device_status_null(lib):
    assert lib.attn_device_status(None, 0) == 1


def test_binding_raises_without_cuda_tensors():
    import torch
    q = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        ap.attn_fwd(q, q, q, False, 0.125)


def test_chunk_scan_rejects_bad_arguments_on_host(lib):
    """chunk_scan_fwd validates before any CUDA call (fake pointers)."""
    f = lib.chunk_scan_fwd
    good = dict(B=1, L=256, H=4, G=1, P=64, Q=256)

    def call(cb=A, da=A, dt=A, x=A, out=A, **kw):
        d = dict(good, **kw)
        return f(cb, da, dt, x, out, d["B"], d["L"], d["H"], d["G"], d["P"], d["Q"], None)

    assert call(cb=0) == 1                      # null pointer
    assert call(L=300) == 1                     # L not a multiple of Q
    assert call(H=3, G=2) == 1                  # H not a multiple of G
    assert call(B=0) == 1
    assert call(P=128) == 2                     # head width other than 64
    assert call(Q=64, L=256) == 2               # chunk other than 128 or 256
    assert call(x=A + 8) == 3                   # misaligned


def test_chunk_scan_host_entry_rejects_before_queuing(lib):
    """chunk_scan_fwd_host: null host buffers, then chunk_scan_fwd's rules on
    the device buffers (fake pointers), all on the host."""
    f = lib.chunk_scan_fwd_host
    dims = [1, 256, 4, 1, 64, 256, None]
    for i in range(5):
        host = [A] * 5
        host[i] = None
        assert f(*host, *([A] * 5), *dims) == 1
    assert f(*([A] * 5), A, A, None, A, A, *dims) == 1                  # null device buffer
    assert f(*([A] * 5), *([A] * 5), 1, 300, 4, 1, 64, 256, None) == 1  # L not a multiple of Q
    assert f(*([A] * 5), *([A] * 5), 1, 256, 4, 1, 128, 256, None) == 2  # P = 128
    assert f(*([A] * 5), A, A, A, A + 8, A, *dims) == 3                 # misaligned x


def test_bwd_workspace_bytes(lib):
    """4 (D + 2) bytes per query row, rows padded to a multiple of 128 per
    (batch, kv-head) group: the per-row vectors and the fp32 dQ accumulator."""
    R = (8 // 2) * 300                      # rows of a group
    Rp = (R + 127) // 128 * 128
    for D in (64, 128):
        assert lib.attn_bwd_workspace_bytes(2, 8, 2, 300, D) == (D + 2) * 2 * 2 * Rp * 4
    assert lib.attn_bwd_workspace_bytes(2, 8, 2, 300, 96) == 0
    assert lib.attn_bwd_workspace_bytes(2, 8, 3, 300, 128) == 0
    assert lib.attn_bwd_workspace_bytes(0, 8, 2, 300, 128) == 0


def test_bwd_entries_reject_before_launch(lib):
    """attn_bwd_deterministic and the backward's timeout hook share
    attn_bwd's checks; every call here fails them (fake device addresses,
    never dereferenced)."""
    ws_bytes = lib.attn_bwd_workspace_bytes(1, 4, 2, 128, 128)
    dims = [1, 4, 2, 128, 128, 128, 0, ctypes.c_float(0.1)]
    bufs = [A] * 9
    no_dout = [A] * 9
    no_dout[5] = None
    assert lib.attn_bwd_deterministic(*no_dout, A, ws_bytes, *dims, None) == 1
    assert lib.attn_bwd_deterministic(*bufs, A, ws_bytes - 1, *dims, None) == 1
    assert lib.attn_bwd_deterministic(*bufs, A + 16, ws_bytes, *dims, None) == 3
    bad_d = [1, 4, 2, 128, 128, 96, 0, ctypes.c_float(0.1)]
    assert lib.attn_bwd_deterministic(*bufs, A, ws_bytes, *bad_d, None) == 2
    assert lib.attn_bwd_timeout_test(*bufs, A, ws_bytes, *dims, -1, 20_000_000, None) == 1
    assert lib.attn_bwd_timeout_test(*bufs, A, ws_bytes, *dims, 1, 10, None) == 1
    assert lib.attn_bwd_timeout_test(*bufs, A, ws_bytes, *dims, 1, 10**10, None) == 1
    assert lib.attn_bwd_timeout_test(*bufs, A, ws_bytes, *bad_d, 1, 20_000_000, None) == 2
