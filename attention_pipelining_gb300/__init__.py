"""GB300 (sm_103a) fused attention forward -- Python binding of libattn_gb300.so.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/attn.h``.  PyTorch supplies
device memory and the current CUDA stream.  There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.

    o, lse = attn_fwd(q, k, v, causal, scale)

q [B, H_q, S_q, D], k and v [B, H_kv, S_kv, D]: contiguous bf16 CUDA tensors,
D in {64, 128}, H_q a multiple of H_kv.  o is bf16 [B, H_q, S_q, D], lse is
fp32 [B, H_q, S_q] (natural log).
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as _LIB_PATH, build as _build_lib

__all__ = ["attn_fwd", "attn_fwd_out", "attn_fwd_host", "attn_fwd_trace", "attn_fwd_splitkv",
           "splitkv_default_splits", "attn_bwd", "attn_bwd_host", "bwd_workspace_bytes",
           "chunk_scan", "chunk_scan_host", "selftest_qk", "selftest_pv", "device_status", "status_string",
           "lib_path", "build", "AttnError", "STATUS"]

STATUS = {
    0: "ATTN_OK",
    1: "ATTN_ERR_INVALID_ARG",
    2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_MISALIGNED",
    4: "ATTN_ERR_CUDA",
    5: "ATTN_ERR_TIMEOUT",
}

# every entry point of include/attn.h and include/attn_selftest.h
EXPORTS = ["attn_fwd", "attn_fwd_host", "attn_status_string", "attn_device_status",
           "attn_version", "attn_selftest_qk", "attn_selftest_pv", "attn_fwd_trace",
           "attn_fwd_timeout_test", "attn_fwd_tail_timeout_test", "attn_fwd_tail_pairs",
           "attn_fwd_splitkv", "attn_splitkv_workspace_bytes",
           "attn_splitkv_default_splits", "attn_fwd_splitkv_noalloc",
           "attn_splitkv_noalloc_capacity", "attn_bwd", "attn_bwd_deterministic",
           "attn_bwd_workspace_bytes", "attn_bwd_timeout_test",
           "attn_bwd_host", "chunk_scan_fwd", "chunk_scan_fwd_host"]


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({status_string(code)})")


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is not built; run attention_pipelining_gb300._build.build() "
            "(needs nvcc) -- there is no fallback implementation")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, vp]
    lib.attn_fwd.restype = ci
    lib.attn_fwd_host.argtypes = [vp] * 10 + [ci] * 7 + [cf, vp]
    lib.attn_fwd_host.restype = ci
    lib.attn_status_string.argtypes = [ci]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_device_status.argtypes = [ctypes.POINTER(ci), ci]
    lib.attn_device_status.restype = ci
    lib.attn_version.argtypes = []
    lib.attn_version.restype = ci
    lib.attn_selftest_qk.argtypes = [vp, vp, vp, ci, vp]
    lib.attn_selftest_qk.restype = ci
    lib.attn_selftest_pv.argtypes = [vp, vp, vp, ci, vp]
    lib.attn_selftest_pv.restype = ci
    lib.attn_fwd_trace.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, vp, ci, ci, vp]
    lib.attn_fwd_trace.restype = ci
    lib.attn_fwd_timeout_test.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf, ci,
                                          ctypes.c_ulonglong, vp]
    lib.attn_fwd_timeout_test.restype = ci
    lib.attn_fwd_tail_timeout_test.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf,
                                               ctypes.c_ulonglong, vp]
    lib.attn_fwd_tail_timeout_test.restype = ci
    lib.attn_fwd_tail_pairs.argtypes = [ci] * 7
    lib.attn_fwd_tail_pairs.restype = ci
    lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                     ci, ci, ci, ci, ci, ci, ci, cf, ci, vp]
    lib.attn_fwd_splitkv.restype = ci
    lib.attn_splitkv_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
    lib.attn_splitkv_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_splitkv_default_splits.argtypes = [ci, ci, ci, ci, ci, ci]
    lib.attn_splitkv_default_splits.restype = ci
    lib.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, cf,
                                             ci, vp]
    lib.attn_fwd_splitkv_noalloc.restype = ci
    lib.attn_splitkv_noalloc_capacity.argtypes = []
    lib.attn_splitkv_noalloc_capacity.restype = ctypes.c_size_t
    lib.attn_bwd.argtypes = [vp] * 10 + [ctypes.c_size_t] + [ci] * 7 + [cf, vp]
    lib.attn_bwd.restype = ci
    lib.attn_bwd_deterministic.argtypes = [vp] * 10 + [ctypes.c_size_t] + [ci] * 7 + [cf, vp]
    lib.attn_bwd_deterministic.restype = ci
    lib.attn_bwd_timeout_test.argtypes = [vp] * 10 + [ctypes.c_size_t] + [ci] * 7 + [cf, ci,
                                          ctypes.c_ulonglong, vp]
    lib.attn_bwd_timeout_test.restype = ci
    lib.attn_bwd_host.argtypes = [vp] * 19 + [ctypes.c_size_t] + [ci] * 7 + [cf, vp]
    lib.attn_bwd_host.restype = ci
    lib.attn_bwd_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.chunk_scan_fwd.argtypes = [vp] * 5 + [ci] * 6 + [vp]
    lib.chunk_scan_fwd.restype = ci
    lib.chunk_scan_fwd_host.argtypes = [vp] * 10 + [ci] * 6 + [vp]
    lib.chunk_scan_fwd_host.restype = ci
    _lib = lib
    return lib


def build(force: bool = False) -> str:
    """Compile the CUDA library (nvcc, sm_103a) if needed and load it."""
    global _lib
    path = _build_lib(force=force)
    _lib = None
    _load()
    return path


def status_string(code: int) -> str:
    return _load().attn_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != 0:
        raise AttnError(code, where)


def _stream_handle(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_inputs(q, k, v):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D [B, H, S, D] tensor")
    if k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")


def attn_fwd_out(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """Writes O and LSE into caller-allocated ``o`` (bf16) and ``lse`` (fp32)."""
    _check_inputs(q, k, v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    _check(_load().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale),
                            _stream_handle(stream)), "attn_fwd")


def attn_fwd(q, k, v, causal: bool, scale: float, stream=None):
    """Fused attention forward; returns (o, lse) allocated on q's device."""
    import torch
    _check_inputs(q, k, v)
    B, Hq, Sq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    attn_fwd_out(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def attn_fwd_host(q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev, o_dev, lse_dev,
                  causal: bool, scale: float, stream=None) -> None:
    """Host-buffer entry: copies q/k/v (host, ideally pinned) into the device
    buffers, runs the kernel, copies o/lse back, all queued on ``stream``."""
    B, Hq, Sq, D = q_dev.shape
    Hkv, Skv = k_dev.shape[1], k_dev.shape[2]
    _check(_load().attn_fwd_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(),
                                 o_host.data_ptr(), lse_host.data_ptr(), q_dev.data_ptr(),
                                 k_dev.data_ptr(), v_dev.data_ptr(), o_dev.data_ptr(),
                                 lse_dev.data_ptr(), B, Hq, Hkv, Sq, Skv, D, int(bool(causal)),
                                 float(scale), _stream_handle(stream)), "attn_fwd_host")


TRACE_EVENTS = ["sm0_wake", "sm0_loaded", "sm0_done", "sm1_wake", "sm1_loaded", "sm1_done",
                "mma_pv0", "mma_s0", "mma_pv1", "mma_s1", "corr0", "corr1", "load_k", "load_v",
                "epilogue", "end", "mma_pv0_begin", "mma_s0_begin", "mma_pv1_begin", "mma_s1_begin"]
MAX_TRACE_BLOCKS = 128  # KV blocks the trace instantiation records per event, at most


def attn_fwd_trace(q, k, v, causal: bool, scale: float, ctas: int = 4, blocks: int | None = None,
                   stream=None):
    """Runs the trace instantiation; returns (o, lse, trace) where trace is an
    int64 CPU tensor [ctas, 20, blocks] of SM clock cycles (0 = no event), for the
    first tile of each traced CTA; blocks <= MAX_TRACE_BLOCKS."""
    import torch
    _check_inputs(q, k, v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    if blocks is None:
        blocks = min((Skv + 127) // 128, MAX_TRACE_BLOCKS)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    tr = torch.zeros((ctas, len(TRACE_EVENTS), blocks), dtype=torch.int64, device=q.device)
    _check(_load().attn_fwd_trace(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, Hq, Hkv, Sq, Skv, D, int(bool(causal)),
                                  float(scale), tr.data_ptr(), ctas, blocks,
                                  _stream_handle(stream)), "attn_fwd_trace")
    torch.cuda.synchronize(q.device)
    return o, lse, tr.cpu()


def splitkv_default_splits(B, H_q, H_kv, S_q, S_kv, causal) -> int:
    return int(_load().attn_splitkv_default_splits(B, H_q, H_kv, S_q, S_kv, int(bool(causal))))


def attn_fwd_splitkv(q, k, v, causal: bool, scale: float, num_splits: int = 0, workspace=None,
                     stream=None):
    """Split-KV forward; returns (o, lse).  ``workspace``: optional uint8 CUDA
    tensor of at least attn_splitkv_workspace_bytes bytes (allocated if None)."""
    import torch
    _check_inputs(q, k, v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    splits = num_splits if num_splits > 0 else splitkv_default_splits(B, Hq, Hkv, Sq, Skv, causal)
    nbytes = int(_load().attn_splitkv_workspace_bytes(B, Hq, Sq, D, splits))
    if nbytes == 0:
        raise AttnError(1, "attn_splitkv_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(_load().attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                    B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale),
                                    int(splits), _stream_handle(stream)), "attn_fwd_splitkv")
    return o, lse


def bwd_workspace_bytes(B, H_q, H_kv, S_q, D) -> int:
    return int(_load().attn_bwd_workspace_bytes(B, H_q, H_kv, S_q, D))


def attn_bwd(q, k, v, o, lse, dout, causal: bool, scale: float, workspace=None, out=None,
             stream=None, deterministic: bool = False):
    """Backward of attn_fwd: returns (dq, dk, dv) for the upstream gradient
    ``dout``, given the forward's ``o`` and ``lse``.  ``workspace``: optional
    uint8 CUDA tensor of at least bwd_workspace_bytes(...) bytes (allocated if
    None); ``out``: optional (dq, dk, dv) to write into.  ``deterministic``
    calls attn_bwd_deterministic (bit-reproducible dQ, see attn.h)."""
    import torch
    _check_inputs(q, k, v)
    for name, t, ref in (("o", o, q), ("dout", dout, q)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.shape != ref.shape \
                or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Sq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H_q, S_q] tensor")
    nbytes = bwd_workspace_bytes(B, Hq, Hkv, Sq, D)
    if nbytes == 0:
        raise AttnError(1, "attn_bwd_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = out
    lib = _load()
    fn = lib.attn_bwd_deterministic if deterministic else lib.attn_bwd
    _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
              lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
              dv.data_ptr(), workspace.data_ptr(), workspace.numel(),
              B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale),
              _stream_handle(stream)), "attn_bwd_deterministic" if deterministic else "attn_bwd")
    return dq, dk, dv


def attn_bwd_host(q_host, k_host, v_host, o_host, lse_host, dout_host, dq_host, dk_host, dv_host,
                  q_dev, k_dev, v_dev, o_dev, lse_dev, dout_dev, dq_dev, dk_dev, dv_dev,
                  causal: bool, scale: float, workspace, stream=None) -> None:
    """Host-buffer backward: copies q, k, v, o, lse, dout (host, ideally
    pinned) into the device buffers, runs attn_bwd with ``workspace`` (a uint8
    CUDA tensor of at least bwd_workspace_bytes(...) bytes), copies dq, dk, dv
    back, all queued on ``stream``."""
    B, Hq, Sq, D = q_host.shape
    Hkv, Skv = k_host.shape[1], k_host.shape[2]
    ts = (q_host, k_host, v_host, o_host, lse_host, dout_host, dq_host, dk_host, dv_host,
          q_dev, k_dev, v_dev, o_dev, lse_dev, dout_dev, dq_dev, dk_dev, dv_dev)
    _check(_load().attn_bwd_host(*(t.data_ptr() for t in ts), workspace.data_ptr(),
                                 workspace.numel(), B, Hq, Hkv, Sq, Skv, D, int(bool(causal)),
                                 float(scale), _stream_handle(stream)), "attn_bwd_host")


def chunk_scan(cb, dA_cs, dt, x, out=None, stream=None):
    """Mamba2 chunk scan (intra-chunk part, include/chunk_scan.h): returns out
    [B, L, H, P] bf16 for cb [B, L/Q, G, Q, Q], dA_cs and dt [B, H, L/Q, Q]
    (float32) and x [B, L, H, P] (bf16), all contiguous CUDA tensors."""
    import torch
    for name, t, dt_ in (("cb", cb, torch.float32), ("dA_cs", dA_cs, torch.float32),
                         ("dt", dt, torch.float32), ("x", x, torch.bfloat16)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dt_ \
                or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA {dt_} tensor")
    B, L, H, P = x.shape
    Bc, nch, G, Q, Q2 = cb.shape
    if Bc != B or Q != Q2 or nch * Q != L or tuple(dA_cs.shape) != (B, H, nch, Q) \
            or tuple(dt.shape) != (B, H, nch, Q):
        raise ValueError("shape mismatch between cb, dA_cs, dt and x")
    if out is None:
        out = torch.empty_like(x)
    _check(_load().chunk_scan_fwd(cb.data_ptr(), dA_cs.data_ptr(), dt.data_ptr(), x.data_ptr(),
                                  out.data_ptr(), B, L, H, G, P, Q, _stream_handle(stream)),
           "chunk_scan_fwd")
    return out


def chunk_scan_host(cb_host, dA_cs_host, dt_host, x_host, out_host, cb_dev, dA_cs_dev, dt_dev,
                    x_dev, out_dev, stream=None) -> None:
    """Host-buffer chunk scan: copies cb, dA_cs, dt, x (host, ideally pinned)
    into the device buffers, runs chunk_scan_fwd, copies out back, all queued
    on ``stream``."""
    B, L, H, P = x_host.shape
    G, Q = cb_host.shape[2], cb_host.shape[3]
    ts = (cb_host, dA_cs_host, dt_host, x_host, out_host, cb_dev, dA_cs_dev, dt_dev, x_dev,
          out_dev)
    _check(_load().chunk_scan_fwd_host(*(t.data_ptr() for t in ts), B, L, H, G, P, Q,
                                       _stream_handle(stream)), "chunk_scan_fwd_host")


def fwd_timeout_test(q, k, v, causal: bool, scale: float, drop_block: int,
                     wait_budget_ns: int = 20_000_000, stream=None):
    """Test hook: runs the forward with one P-ready signal withheld at KV block
    ``drop_block`` so the kernel's bounded wait runs out (see attn_testing.h).
    Returns (o, lse); the device status word then reads ATTN_ERR_TIMEOUT."""
    import torch
    _check_inputs(q, k, v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(_load().attn_fwd_timeout_test(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, Hq, Hkv, Sq, Skv, D, int(bool(causal)),
                                         float(scale), int(drop_block), int(wait_budget_ns),
                                         _stream_handle(stream)), "attn_fwd_timeout_test")
    return o, lse


def bwd_timeout_test(q, k, v, o, lse, dout, causal: bool, scale: float, drop_item: int,
                     wait_budget_ns: int = 20_000_000, stream=None):
    """Test hook: runs attn_bwd with one "P^T, dS^T stored" signal withheld
    at work item ``drop_item`` of every dK/dV CTA, so the issuer's bounded
    wait runs out (see attn_testing.h).  Returns (dq, dk, dv); the device
    status word then reads ATTN_ERR_TIMEOUT."""
    import torch
    _check_inputs(q, k, v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    ws = torch.empty(bwd_workspace_bytes(B, Hq, Hkv, Sq, D), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _check(_load().attn_bwd_timeout_test(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                                         dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), ws.numel(),
                                         B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale),
                                         int(drop_item), int(wait_budget_ns),
                                         _stream_handle(stream)), "attn_bwd_timeout_test")
    return dq, dk, dv


def fwd_tail_timeout_test(q, k, v, causal: bool, scale: float,
                          wait_budget_ns: int = 20_000_000, stream=None):
    """Test hook: runs the forward's split-tail launch with no CTA of a pair
    sending its staged partial, so the bounded cluster waits for it run out
    (see attn_testing.h).  Returns (o, lse); the device status word
    then reads ATTN_ERR_TIMEOUT."""
    import torch
    _check_inputs(q, k, v)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _check(_load().attn_fwd_tail_timeout_test(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                              o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Skv,
                                              D, int(bool(causal)), float(scale),
                                              int(wait_budget_ns), _stream_handle(stream)),
           "attn_fwd_tail_timeout_test")
    return o, lse


def fwd_tail_pairs(B: int, H_q: int, H_kv: int, S_q: int, S_kv: int, D: int, causal: bool) -> int:
    """Tiles attn_fwd splits across CTA pairs for these sizes on the current
    device (0: none; -1: invalid sizes or no device)."""
    return int(_load().attn_fwd_tail_pairs(B, H_q, H_kv, S_q, S_kv, D, int(bool(causal))))


def selftest_qk(q, k):
    """s = q k^T ([128, D] bf16 each) through TMA + tcgen05, fp32 [128, 128]."""
    import torch
    s = torch.empty((128, 128), dtype=torch.float32, device=q.device)
    _check(_load().attn_selftest_qk(q.data_ptr(), k.data_ptr(), s.data_ptr(), q.shape[1],
                                    _stream_handle(None)), "attn_selftest_qk")
    return s


def selftest_pv(p, v):
    """o = p v (p [128, 128] bf16 via tensor memory, v [128, D] bf16), fp32 [128, D]."""
    import torch
    o = torch.empty((128, v.shape[1]), dtype=torch.float32, device=v.device)
    _check(_load().attn_selftest_pv(p.data_ptr(), v.data_ptr(), o.data_ptr(), v.shape[1],
                                    _stream_handle(None)), "attn_selftest_pv")
    return o


def device_status(reset: bool = True) -> int:
    """The device-side status word (0, or 5 = a kernel wait timed out)."""
    st = ctypes.c_int(0)
    _check(_load().attn_device_status(ctypes.byref(st), int(bool(reset))), "attn_device_status")
    return st.value
