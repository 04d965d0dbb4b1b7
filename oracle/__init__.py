"""fp64 CPU oracle for the attention forward and backward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package.  The CUDA product path never touches
it: the two share no code, header, table or helper.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over output
rows).  It is the definition written out, following "PipeThreader:
Software-Defined Pipelining for Efficient DNN Execution", section A2,
paragraph "FlashAttention-3" and Fig. 7 (acc_s = Q K^T -> Softmax -> P ->
P V = O), with the readings listed at the top of the C file (scale before
the mask, top-left causal mask j <= i, grouped heads h // (H_q / H_kv),
natural-log LSE, [B, H, S, D] layout).

The backward (``attn_bwd_oracle.c``, its own library) is the chain rule
through that definition: dQ, dK, dV of L = sum(O * dO), with D_i = dO_i . O_i
and dS = P (dP - D); it also takes fp64 inputs so finite differences of the
forward can check it.

The Mamba2 chunk scan (``chunk_scan_oracle.c``, its own library) is the
intra-chunk sum out[m] = sum_{k <= m} cb[m, k] exp(dA_cs[m] - dA_cs[k]) dt[k]
x[k], written out row by row.

This module only builds the shared libraries and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_BWD_SRC = os.path.join(_HERE, "attn_bwd_oracle.c")
_BWD_LIB = os.path.join(_HERE, "libbwd_oracle.so")
_CS_SRC = os.path.join(_HERE, "chunk_scan_oracle.c")
_CS_LIB = os.path.join(_HERE, "libchunk_scan_oracle.so")
_default = None
_bwd_default = None
_cs_default = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c, attn_bwd_oracle.c and chunk_scan_oracle.c into
    liboracle.so, libbwd_oracle.so and libchunk_scan_oracle.so next to them
    (gcc, -O2, OpenMP); returns the first."""
    for src, lib in ((_SRC, _LIB), (_BWD_SRC, _BWD_LIB), (_CS_SRC, _CS_LIB)):
        if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
            compile_source(src, lib)
    return _LIB


def compile_source(src: str, out: str) -> str:
    """gcc a C file with the oracle's exported functions into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    ci, cd = ctypes.c_int, ctypes.c_double
    lib.oracle_attn_fwd.argtypes = [u16p, u16p, u16p, f64p, f64p,
                                    ci, ci, ci, ci, ci, ci, ci, cd]
    lib.oracle_attn_fwd.restype = ci
    lib.oracle_attn_rows.argtypes = [u16p, u16p, u16p, i64p, ctypes.c_int64,
                                     f64p, f64p, ci, ci, ci, ci, ci, ci, ci, cd]
    lib.oracle_attn_rows.restype = ci
    lib.oracle_attn_probs.argtypes = [u16p, u16p, u16p, f64p, f64p, f64p,
                                      ci, ci, ci, ci, ci, ci, ci, cd]
    lib.oracle_attn_probs.restype = ci
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ci
    return lib


def _bits(x) -> np.ndarray:
    """bf16 input as a contiguous uint16 bit array.

    Accepts a torch.bfloat16 tensor (any device; copied to the CPU) or a numpy
    uint16 array of bf16 bit patterns.
    """
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bf16 bit patterns")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("oracle inputs must be bfloat16")
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _dims(q, k, v):
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return B, Hq, Hkv, Sq, Skv, D


class Oracle:
    """Handle on one compiled copy of the oracle library."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _bind(path)

    def attn_fwd(self, q, k, v, causal: bool, scale: float):
        """O [B,H_q,S_q,D] and LSE [B,H_q,S_q], both float64 numpy arrays."""
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        o = np.empty((B, Hq, Sq, D), np.float64)
        lse = np.empty((B, Hq, Sq), np.float64)
        rc = self.lib.oracle_attn_fwd(
            _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
            _p(o, ctypes.c_double), _p(lse, ctypes.c_double),
            B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_fwd rejected the arguments (rc={rc})")
        return o, lse

    def attn_rows(self, q, k, v, rows, causal: bool, scale: float):
        """O and LSE for the flat row indices ``rows`` into [B, H_q, S_q].

        Returns (o_rows [n, D], lse_rows [n]) as float64 numpy arrays.
        """
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.empty((r.size, D), np.float64)
        lse = np.empty((r.size,), np.float64)
        rc = self.lib.oracle_attn_rows(
            _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
            _p(r, ctypes.c_int64), r.size, _p(o, ctypes.c_double), _p(lse, ctypes.c_double),
            B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_rows rejected the arguments (rc={rc})")
        return o, lse

    def attn_probs(self, q, k, v, causal: bool, scale: float):
        """P [B,H_q,S_q,S_kv], O and LSE as float64 numpy arrays (tiny sizes)."""
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        qb, kb, vb = _bits(q), _bits(k), _bits(v)
        p = np.empty((B, Hq, Sq, Skv), np.float64)
        o = np.empty((B, Hq, Sq, D), np.float64)
        lse = np.empty((B, Hq, Sq), np.float64)
        rc = self.lib.oracle_attn_probs(
            _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
            _p(p, ctypes.c_double), _p(o, ctypes.c_double), _p(lse, ctypes.c_double),
            B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_probs rejected the arguments (rc={rc})")
        return p, o, lse

    def num_threads(self) -> int:
        """OpenMP threads the oracle runs on."""
        return int(self.lib.oracle_num_threads())


def default() -> Oracle:
    """The oracle built from attn_oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def attn_fwd(q, k, v, causal: bool, scale: float):
    return default().attn_fwd(q, k, v, causal, scale)


def attn_rows(q, k, v, rows, causal: bool, scale: float):
    return default().attn_rows(q, k, v, rows, causal, scale)


def attn_probs(q, k, v, causal: bool, scale: float):
    return default().attn_probs(q, k, v, causal, scale)


def num_threads() -> int:
    return default().num_threads()


# ---------------------------------------------------------------- backward


def _bind_bwd(path: str):
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    ci, cd = ctypes.c_int, ctypes.c_double
    dims = [ci, ci, ci, ci, ci, ci, ci, cd]
    lib.oracle_attn_bwd.argtypes = [u16p, u16p, u16p, u16p, f64p, f64p, f64p] + dims
    lib.oracle_attn_bwd_f64.argtypes = [f64p, f64p, f64p, f64p, f64p, f64p, f64p] + dims
    lib.oracle_attn_fwd_f64.argtypes = [f64p, f64p, f64p, f64p, f64p] + dims
    lib.oracle_attn_bwd_dq_rows.argtypes = [u16p, u16p, u16p, u16p, i64p, ctypes.c_int64,
                                            f64p] + dims
    lib.oracle_attn_bwd_dkv_rows.argtypes = [u16p, u16p, u16p, u16p, i64p, ctypes.c_int64,
                                             f64p, f64p] + dims
    for f in ("oracle_attn_bwd", "oracle_attn_bwd_f64", "oracle_attn_fwd_f64",
              "oracle_attn_bwd_dq_rows", "oracle_attn_bwd_dkv_rows"):
        getattr(lib, f).restype = ci
    return lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


class BwdOracle:
    """Handle on one compiled copy of the backward oracle library."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _bind_bwd(path)

    def attn_bwd(self, q, k, v, dout, causal: bool, scale: float):
        """dQ [B,H_q,S_q,D], dK and dV [B,H_kv,S_kv,D] (float64) for bf16 inputs."""
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        if tuple(dout.shape) != tuple(q.shape):
            raise ValueError("dout must have q's shape")
        qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
        dq = np.empty((B, Hq, Sq, D), np.float64)
        dk = np.empty((B, Hkv, Skv, D), np.float64)
        dv = np.empty((B, Hkv, Skv, D), np.float64)
        rc = self.lib.oracle_attn_bwd(
            _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
            _p(db, ctypes.c_uint16), _p(dq, ctypes.c_double), _p(dk, ctypes.c_double),
            _p(dv, ctypes.c_double), B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd rejected the arguments (rc={rc})")
        return dq, dk, dv

    def attn_bwd_f64(self, q, k, v, dout, causal: bool, scale: float):
        """The same for float64 numpy inputs (no bf16 rounding)."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        if dout.shape != q.shape:
            raise ValueError("dout must have q's shape")
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
        rc = self.lib.oracle_attn_bwd_f64(
            _p(q, ctypes.c_double), _p(k, ctypes.c_double), _p(v, ctypes.c_double),
            _p(dout, ctypes.c_double), _p(dq, ctypes.c_double), _p(dk, ctypes.c_double),
            _p(dv, ctypes.c_double), B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_f64 rejected the arguments (rc={rc})")
        return dq, dk, dv

    def attn_fwd_f64(self, q, k, v, causal: bool, scale: float):
        """Forward O and LSE for float64 numpy inputs."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        o = np.empty_like(q)
        lse = np.empty((B, Hq, Sq), np.float64)
        rc = self.lib.oracle_attn_fwd_f64(
            _p(q, ctypes.c_double), _p(k, ctypes.c_double), _p(v, ctypes.c_double),
            _p(o, ctypes.c_double), _p(lse, ctypes.c_double),
            B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_fwd_f64 rejected the arguments (rc={rc})")
        return o, lse

    def dq_rows(self, q, k, v, dout, rows, causal: bool, scale: float):
        """dQ of the flat query rows ``rows`` into [B, H_q, S_q]: [n, D] float64."""
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        if tuple(dout.shape) != tuple(q.shape):
            raise ValueError("dout must have q's shape")
        qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.empty((r.size, D), np.float64)
        rc = self.lib.oracle_attn_bwd_dq_rows(
            _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
            _p(db, ctypes.c_uint16), _p(r, ctypes.c_int64), r.size, _p(out, ctypes.c_double),
            B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_dq_rows rejected the arguments (rc={rc})")
        return out

    def dkv_rows(self, q, k, v, dout, rows, causal: bool, scale: float):
        """dK and dV of the flat key rows ``rows`` into [B, H_kv, S_kv]: two [n, D]."""
        B, Hq, Hkv, Sq, Skv, D = _dims(q, k, v)
        if tuple(dout.shape) != tuple(q.shape):
            raise ValueError("dout must have q's shape")
        qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        dk = np.empty((r.size, D), np.float64)
        dv = np.empty((r.size, D), np.float64)
        rc = self.lib.oracle_attn_bwd_dkv_rows(
            _p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
            _p(db, ctypes.c_uint16), _p(r, ctypes.c_int64), r.size, _p(dk, ctypes.c_double),
            _p(dv, ctypes.c_double), B, Hq, Hkv, Sq, Skv, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_dkv_rows rejected the arguments (rc={rc})")
        return dk, dv


def bwd_default() -> BwdOracle:
    """The backward oracle built from attn_bwd_oracle.c (compiled on first use)."""
    global _bwd_default
    if _bwd_default is None:
        build()
        _bwd_default = BwdOracle(_BWD_LIB)
    return _bwd_default


def attn_bwd(q, k, v, dout, causal: bool, scale: float):
    return bwd_default().attn_bwd(q, k, v, dout, causal, scale)


# ---------------------------------------------------------------- chunk scan


def _bind_cs(path: str):
    lib = ctypes.CDLL(path)
    f32p = ctypes.POINTER(ctypes.c_float)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    ci = ctypes.c_int
    dims = [ci] * 6
    lib.oracle_chunk_scan.argtypes = [f32p, f32p, f32p, u16p, f64p] + dims
    lib.oracle_chunk_scan.restype = ci
    lib.oracle_chunk_scan_rows.argtypes = [f32p, f32p, f32p, u16p, i64p, ctypes.c_int64,
                                           f64p] + dims
    lib.oracle_chunk_scan_rows.restype = ci
    return lib


def _f32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


class ChunkScanOracle:
    """Handle on one compiled copy of the chunk-scan oracle library."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _bind_cs(path)

    @staticmethod
    def _dims(cb, dA_cs, dt, x):
        B, L, H, P = x.shape
        Bc, nch, G, Q, Q2 = cb.shape
        if Bc != B or Q != Q2 or nch * Q != L or tuple(dA_cs.shape) != (B, H, nch, Q) \
                or tuple(dt.shape) != (B, H, nch, Q):
            raise ValueError(f"shape mismatch cb{tuple(cb.shape)} dA_cs{tuple(dA_cs.shape)} "
                             f"dt{tuple(dt.shape)} x{tuple(x.shape)}")
        return B, L, H, G, P, Q

    def chunk_scan(self, cb, dA_cs, dt, x):
        """out [B, L, H, P] float64 for cb, dA_cs, dt (float32) and x (bf16)."""
        B, L, H, G, P, Q = self._dims(cb, dA_cs, dt, x)
        c, a, d, xb = _f32(cb), _f32(dA_cs), _f32(dt), _bits(x)
        out = np.empty((B, L, H, P), np.float64)
        rc = self.lib.oracle_chunk_scan(_p(c, ctypes.c_float), _p(a, ctypes.c_float),
                                        _p(d, ctypes.c_float), _p(xb, ctypes.c_uint16),
                                        _p(out, ctypes.c_double), B, L, H, G, P, Q)
        if rc != 0:
            raise ValueError(f"oracle_chunk_scan rejected the arguments (rc={rc})")
        return out

    def rows(self, cb, dA_cs, dt, x, rows):
        """Output rows (flat indices into [B, L, H]): [n, P] float64."""
        B, L, H, G, P, Q = self._dims(cb, dA_cs, dt, x)
        c, a, d, xb = _f32(cb), _f32(dA_cs), _f32(dt), _bits(x)
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        out = np.empty((r.size, P), np.float64)
        rc = self.lib.oracle_chunk_scan_rows(_p(c, ctypes.c_float), _p(a, ctypes.c_float),
                                             _p(d, ctypes.c_float), _p(xb, ctypes.c_uint16),
                                             _p(r, ctypes.c_int64), r.size,
                                             _p(out, ctypes.c_double), B, L, H, G, P, Q)
        if rc != 0:
            raise ValueError(f"oracle_chunk_scan_rows rejected the arguments (rc={rc})")
        return out


def chunk_scan_default() -> ChunkScanOracle:
    """The chunk-scan oracle built from chunk_scan_oracle.c (compiled on first use)."""
    global _cs_default
    if _cs_default is None:
        build()
        _cs_default = ChunkScanOracle(_CS_LIB)
    return _cs_default
