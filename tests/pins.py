"""Checks that pin the fp64 oracle to facts fixed by the definition of attention.

Each ``pin_*`` takes an oracle handle (``oracle.Oracle``) and returns a list of
failure strings (empty = the pin holds).  They are written this way so that the
same checks can run against copies of the oracle with a planted mistake
(tests/test_oracle_mutants.py): every plausible mistake must trip one of them.

The definition pinned here ("PipeThreader: Software-Defined Pipelining for
Efficient DNN Execution", section A2, paragraph "FlashAttention-3", Fig. 7):
acc_s = Q K^T (times scale), P = softmax(acc_s) over the visible keys,
O = P V; plus LSE = log sum exp of the scaled scores.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

from attention_pipelining_gb300.synthetic import make_qkv


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _visible(i: int, S_kv: int, causal: bool) -> int:
    return min(i + 1, S_kv) if causal else S_kv


SHAPES = [
    # B, H_q, H_kv, S_q, S_kv, D
    (1, 1, 1, 7, 7, 8),
    (2, 4, 2, 9, 13, 16),
    (1, 3, 1, 12, 5, 4),
    (2, 2, 2, 16, 16, 32),
]


def pin_row_sums(orc) -> list[str]:
    """Every softmax row sums to 1; masked keys get probability exactly 0."""
    errs = []
    for (B, Hq, Hkv, Sq, Skv, D) in SHAPES:
        for causal in (False, True):
            q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=11)
            p, o, lse = orc.attn_probs(q, k, v, causal, 1.0 / math.sqrt(D))
            dev = np.abs(p.sum(-1) - 1.0).max()
            if not dev <= 1e-14:
                errs.append(f"row sum off by {dev} {B,Hq,Hkv,Sq,Skv,D} causal={causal}")
            if causal:
                i = np.arange(Sq)[:, None]
                j = np.arange(Skv)[None, :]
                masked = np.broadcast_to(j > i, p.shape)
                if np.any(p[masked] != 0.0):
                    errs.append(f"masked probability nonzero {B,Hq,Hkv,Sq,Skv,D}")
            if np.any(p < 0):
                errs.append("negative probability")
    return errs


def pin_ones(orc) -> list[str]:
    """V of all ones gives O of all ones, for any Q, K and mask."""
    errs = []
    for (B, Hq, Hkv, Sq, Skv, D) in SHAPES:
        for causal in (False, True):
            q, k, _ = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=5)
            v = torch.ones((B, Hkv, Skv, D), dtype=torch.bfloat16)
            o, _ = orc.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(D))
            dev = np.abs(o - 1.0).max()
            if not dev <= 1e-14:
                errs.append(f"V=1 gives O off by {dev} {B,Hq,Hkv,Sq,Skv,D} causal={causal}")
    return errs


def pin_single_key(orc) -> list[str]:
    """S_kv = 1: the only key gets probability 1, so O = V_0 and LSE = score_0."""
    errs = []
    for (B, Hq, Hkv, Sq, D) in [(1, 1, 1, 5, 8), (2, 4, 2, 3, 16), (1, 6, 3, 4, 64)]:
        for causal in (False, True):
            scale = 0.37
            q, k, v = make_qkv(B, Hq, Hkv, Sq, 1, D, seed=3)
            o, lse = orc.attn_fwd(q, k, v, causal, scale)
            r = Hq // Hkv
            for b in range(B):
                for h in range(Hq):
                    g = h // r
                    want_o = _f64(v[b, g, 0])
                    if not np.array_equal(o[b, h], np.broadcast_to(want_o, o[b, h].shape)):
                        errs.append(f"S_kv=1: O != V_0 at b={b} h={h}")
                    s0 = scale * (_f64(q[b, h]) @ _f64(k[b, g, 0]))
                    dev = np.abs(lse[b, h] - s0).max()
                    if not dev <= 1e-12 * max(1.0, np.abs(s0).max()):
                        errs.append(f"S_kv=1: LSE off by {dev} at b={b} h={h}")
    return errs


def pin_zero_query(orc) -> list[str]:
    """Q = 0: all visible scores tie, so O_i is the mean of the visible V rows
    (a prefix mean when causal) and LSE_i = ln(number of visible keys)."""
    errs = []
    for (B, Hq, Hkv, Sq, Skv, D) in SHAPES + [(1, 2, 1, 20, 6, 8)]:
        for causal in (False, True):
            _, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=7)
            q = torch.zeros((B, Hq, Sq, D), dtype=torch.bfloat16)
            o, lse = orc.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(D))
            r = Hq // Hkv
            v64 = _f64(v)
            for b in range(B):
                for h in range(Hq):
                    for i in range(Sq):
                        n = _visible(i, Skv, causal)
                        want = v64[b, h // r, :n].mean(axis=0)
                        dev = np.abs(o[b, h, i] - want).max()
                        if not dev <= 1e-13:
                            errs.append(f"Q=0: O off by {dev} at {(b, h, i)} causal={causal}")
                            break
                        if not abs(lse[b, h, i] - math.log(n)) <= 1e-14:
                            errs.append(f"Q=0: LSE {lse[b, h, i]} != ln {n} at {(b, h, i)}")
                            break
    return errs


def pin_permutation(orc) -> list[str]:
    """Non-causal attention is a set function of the (key, value) pairs:
    permuting keys together with their values leaves O and LSE unchanged."""
    errs = []
    for (B, Hq, Hkv, Sq, Skv, D) in SHAPES:
        q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=13)
        perm = torch.randperm(Skv, generator=torch.Generator().manual_seed(1))
        o1, l1 = orc.attn_fwd(q, k, v, False, 1.0 / math.sqrt(D))
        o2, l2 = orc.attn_fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(),
                              False, 1.0 / math.sqrt(D))
        dev = max(np.abs(o1 - o2).max(), np.abs(l1 - l2).max())
        if not dev <= 1e-13:
            errs.append(f"permutation changed the result by {dev} {B,Hq,Hkv,Sq,Skv,D}")
        # and a permutation of keys alone (values fixed) must change it
        o3, _ = orc.attn_fwd(q, k[:, :, perm].contiguous(), v, False, 1.0 / math.sqrt(D))
        if Skv > 1 and np.abs(o1 - o3).max() < 1e-6:
            errs.append("permuting keys without values left O unchanged")
    return errs


def _brute_row(qi, kk, vv, n, scale):
    """Textbook softmax without max subtraction, in plain Python floats."""
    w = []
    for j in range(n):
        s = 0.0
        for d in range(len(qi)):
            s += qi[d] * kk[j][d]
        w.append(math.exp(scale * s))
    tot = math.fsum(w)
    o = [math.fsum(w[j] * vv[j][d] for j in range(n)) / tot for d in range(len(qi))]
    return o, math.log(tot)


def pin_brute_force(orc) -> list[str]:
    """Brute force on 4x4 problems (plus a grouped-head 2:1 case)."""
    errs = []
    for (B, Hq, Hkv, Sq, Skv, D) in [(1, 1, 1, 4, 4, 8), (1, 2, 1, 4, 4, 4), (2, 4, 2, 4, 4, 2)]:
        for causal in (False, True):
            scale = 0.5
            q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=17)
            o, lse = orc.attn_fwd(q, k, v, causal, scale)
            qq, kk, vv = _f64(q).tolist(), _f64(k).tolist(), _f64(v).tolist()
            r = Hq // Hkv
            for b in range(B):
                for h in range(Hq):
                    for i in range(Sq):
                        n = _visible(i, Skv, causal)
                        bo, bl = _brute_row(qq[b][h][i], kk[b][h // r], vv[b][h // r], n, scale)
                        dev = max(np.abs(o[b, h, i] - np.array(bo)).max(), abs(lse[b, h, i] - bl))
                        if not dev <= 1e-13:
                            errs.append(f"brute force off by {dev} at {(b, h, i)} causal={causal}")
    return errs


def pin_powers_of_two(orc) -> list[str]:
    """Closed form: q_i = e_0, k_j = (c_g * j) e_0 for kv head g, scale = ln 2.
    Then the weight of key j is 2^(c_g * j), so with integer values V the output
    is an exact rational (computed here with fractions) and
    LSE_i = ln(sum_{j visible} 2^(c_g j))."""
    errs = []
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 6, 6, 3
    for causal in (False, True):
        q = np.zeros((B, Hq, Sq, D), np.float32)
        q[..., 0] = 1.0
        k = np.zeros((B, Hkv, Skv, D), np.float32)
        v = np.zeros((B, Hkv, Skv, D), np.float32)
        c = [1, 2]
        for g in range(Hkv):
            for j in range(Skv):
                k[0, g, j, 0] = c[g] * j
                for d in range(D):
                    v[0, g, j, d] = ((3 * j + 2 * d + g) % 7) - 3
        o, lse = orc.attn_fwd(_bf16(q), _bf16(k), _bf16(v), causal, math.log(2.0))
        r = Hq // Hkv
        for h in range(Hq):
            g = h // r
            for i in range(Sq):
                n = _visible(i, Skv, causal)
                wts = [Fraction(2) ** (c[g] * j) for j in range(n)]
                tot = sum(wts)
                for d in range(D):
                    want = sum(wts[j] * int(v[0, g, j, d]) for j in range(n)) / tot
                    if not abs(o[0, h, i, d] - float(want)) <= 1e-12:
                        errs.append(f"powers of two: O[{h},{i},{d}]={o[0, h, i, d]} want {float(want)}")
                want_lse = math.log(float(tot))
                if not abs(lse[0, h, i] - want_lse) <= 1e-12 * max(1.0, want_lse):
                    errs.append(f"powers of two: LSE[{h},{i}]={lse[0, h, i]} want {want_lse}")
    return errs


def pin_library_sdpa(orc) -> list[str]:
    """Library special case: torch's float64 CPU scaled_dot_product_attention
    (its causal mask is the top-left lower triangle, grouped heads by
    repeat_interleave) agrees on small and medium shapes."""
    errs = []
    F = torch.nn.functional
    for (B, Hq, Hkv, Sq, Skv, D) in [(1, 2, 2, 33, 33, 16), (2, 8, 2, 64, 64, 64),
                                     (1, 4, 1, 40, 72, 32), (1, 2, 1, 130, 130, 128)]:
        for causal in (False, True):
            scale = 1.0 / math.sqrt(D)
            q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=23)
            o, _ = orc.attn_fwd(q, k, v, causal, scale)
            ref = F.scaled_dot_product_attention(
                q.double(), k.double(), v.double(), is_causal=causal, scale=scale,
                enable_gqa=(Hq != Hkv)).numpy()
            dev = np.abs(o - ref).max()
            if not dev <= 1e-12:
                errs.append(f"torch fp64 SDPA differs by {dev} {B,Hq,Hkv,Sq,Skv,D} causal={causal}")
    return errs


def pin_negative_scale(orc) -> list[str]:
    """A negative scale: torch's float64 SDPA agrees (a library special case),
    and negating the scale is the same as negating the keys (the scores are
    scale * q . k, and negation is exact), bit for bit."""
    import torch.nn.functional as F
    errs = []
    for (B, Hq, Hkv, Sq, Skv, D) in [(1, 2, 2, 33, 47, 16), (2, 4, 2, 40, 40, 32)]:
        for causal in (False, True):
            for scale in (-0.3, -2.5):
                q, k, v = make_qkv(B, Hq, Hkv, Sq, Skv, D, seed=29)
                o, lse = orc.attn_fwd(q, k, v, causal, scale)
                # (an explicit boolean mask: torch's is_causal path gives NaN
                # for a negative scale)
                mask = torch.ones(Sq, Skv, dtype=torch.bool).tril() if causal else None
                ref = F.scaled_dot_product_attention(
                    q.double(), k.double(), v.double(), attn_mask=mask, scale=scale,
                    enable_gqa=(Hq != Hkv)).numpy()
                dev = np.abs(o - ref).max()
                if not dev <= 1e-12:
                    errs.append(f"SDPA differs by {dev} at scale {scale} causal={causal}")
                o2, l2 = orc.attn_fwd(q, (-k).contiguous(), v, causal, -scale)
                if not (np.array_equal(o, o2) and np.array_equal(lse, l2)):
                    errs.append(f"scale {scale} and keys negated with -scale differ")
    return errs


ALL_PINS = [pin_row_sums, pin_ones, pin_single_key, pin_zero_query, pin_permutation,
            pin_brute_force, pin_powers_of_two, pin_library_sdpa, pin_negative_scale]
