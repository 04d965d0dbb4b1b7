"""Per-element error allowance of the CUDA attention backward.

The tolerance is derived from the arithmetic of the GPU path, not from
observed errors.  Every gradient element is a sum of products of bf16 values
(exact in fp32) accumulated in fp32 by the tensor core; what differs from the
exact result are these roundings (u = 2^-8, the unit roundoff of bf16's
8-bit significand; a rounding's relative error is at most u and, spread over
a binade, has standard deviation at most u / sqrt(3)):

  dV_j = sum_i P_ij dO_i         P_ij rounded to bf16 before the GEMM
  dK_j = scale sum_i dS_ij q_i   dS_ij = P_ij (dP_ij - D_i) rounded to bf16,
                                 and D_i = dO_i . O_i uses the forward's bf16 O
  dQ_i = scale sum_j dS_ij k_j   the same dS_ij (recomputed), and the same D_i

D_i's error enters every dS_ij of row i with the same sign (-P_ij dD_i), so
in dQ_i it adds coherently, as dD_i (P k)_i; in dK_j it adds over the rows i
like an independent term.  O's error is its output rounding plus the forward's
own rounding of P before its PV GEMM.  The roundings of different terms are
independent, so each sum's error has standard deviation

  sigma_V^2 = u^2/3 sum_i (P_ij dO_id)^2
  sigma_K^2 = scale^2 [u^2/3 sum_i (dS_ij q_id)^2 + sum_i (P_ij q_id)^2 sigma_Di^2]
  sigma_Q^2 = scale^2 [u^2/3 sum_j (dS_ij k_jd)^2 + sigma_Di^2 (sum_j P_ij k_jd)^2]
  sigma_Di^2 = u^2/3 sum_d dO_id^2 (O_id^2 + sum_j P_ij^2 v_jd^2)

Neglected, each below 2^-14 of sigma at these sizes: the fp32 rounding of the
scores and of the LSE, the exp2 approximation, and the fp32 accumulation
(bounded here by ceil(n / 16) 2^-23 times the root-sum-square of the n terms,
one accumulator rounding per 16-deep MMA step; added to the allowance).

Allowance per element: K_SIGMA * sigma + (accumulation term) + u |ref| (the
output's own rounding to bf16).  With K_SIGMA = 8 a correct kernel exceeds it
with probability below 1e-14 per element (the error is a sum of bounded,
independent terms, lighter-tailed than a normal one).  The scales are computed
here in float64 with torch from q, k, v and dO (the exact softmax), on
whatever device the caller names; they set only the size of the allowance,
the expected values come from the fp64 oracle.
"""
from __future__ import annotations

import math

import numpy as np
import torch

U = 2.0 ** -8          # bf16 unit roundoff
K_SIGMA = 8.0          # allowance in standard deviations of the rounding model
ACC = 2.0 ** -23       # one fp32 accumulator rounding per 16-deep MMA step


def _groups(q, k, v, dout):
    """Row-group views: [Z, R, D] for q and dO, [Z, S_kv, D] for k and v."""
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    rep = Hq // Hkv
    return (q.reshape(B * Hkv, rep * Sq, D), k.reshape(B * Hkv, Skv, D),
            v.reshape(B * Hkv, Skv, D), dout.reshape(B * Hkv, rep * Sq, D), Sq)


def _row_terms(Qr, pos, K, V, dOr, causal, scale):
    """Exact softmax quantities of query rows Qr (positions pos) of one group."""
    s = scale * (Qr @ K.T)
    if causal:
        j = torch.arange(K.shape[0], device=K.device)
        s = s.masked_fill(j[None, :] > pos[:, None], -math.inf)
    P = torch.softmax(s, dim=1)
    O = P @ V
    Dv = (dOr * O).sum(1)
    dS = P * (dOr @ V.T - Dv[:, None])
    sd2 = (U * U / 3) * (dOr * dOr * (O * O + (P * P) @ (V * V))).sum(1)
    return P, dS, sd2


def _acc(n: int) -> float:
    return math.ceil(max(n, 1) / 16) * ACC


def dq_sigma(q, k, v, dout, rows, causal: bool, scale: float, device="cuda", chunk=2048):
    """(sigma, acc) of dQ at the flat query rows ``rows`` of [B, H_q, S_q]:
    two [n, D] float64 numpy arrays."""
    Qg, Kg, Vg, dOg, Sq = (t.to(device, torch.float64) if torch.is_tensor(t) else t
                           for t in _groups(q, k, v, dout))
    R = Qg.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    out_s = np.zeros((rows.size, Qg.shape[2]))
    out_a = np.zeros_like(out_s)
    for z in np.unique(rows // R):
        sel_all = np.nonzero(rows // R == z)[0]
        K = Kg[z]
        for c0 in range(0, sel_all.size, chunk):
            sel = sel_all[c0:c0 + chunk]
            rho = torch.as_tensor(rows[sel] % R, device=device)
            P, dS, sd2 = _row_terms(Qg[z, rho], rho % Sq, K, Vg[z], dOg[z, rho], causal, scale)
            t2 = (dS * dS) @ (K * K)
            var = scale * scale * ((U * U / 3) * t2 + sd2[:, None] * (P @ K) ** 2)
            acc = torch.tensor([_acc(int(c)) for c in (P > 0).sum(1).tolist()],
                               dtype=torch.float64, device=device)[:, None]
            out_s[sel] = torch.sqrt(var).cpu().numpy()
            out_a[sel] = (acc * abs(scale) * torch.sqrt(t2)).cpu().numpy()
    return out_s, out_a


def dkv_sigma(q, k, v, dout, rows, causal: bool, scale: float, device="cuda", chunk=2048):
    """(sigma_K, acc_K, sigma_V, acc_V) at the flat key rows ``rows`` of
    [B, H_kv, S_kv]: four [n, D] float64 numpy arrays."""
    Qg, Kg, Vg, dOg, Sq = (t.to(device, torch.float64) if torch.is_tensor(t) else t
                           for t in _groups(q, k, v, dout))
    Skv, D = Kg.shape[1], Kg.shape[2]
    R = Qg.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    res = [np.zeros((rows.size, D)) for _ in range(4)]
    for z in np.unique(rows // Skv):
        sel = np.nonzero(rows // Skv == z)[0]
        keys = torch.as_tensor(rows[sel] % Skv, device=device)
        vk = torch.zeros((keys.numel(), D), dtype=torch.float64, device=device)
        vq = torch.zeros_like(vk)
        vv = torch.zeros_like(vk)
        cnt = torch.zeros(keys.numel(), dtype=torch.float64, device=device)
        for r0 in range(0, R, chunk):
            Qr = Qg[z, r0:r0 + chunk]
            pos = torch.arange(r0, r0 + Qr.shape[0], device=device) % Sq
            P, dS, sd2 = _row_terms(Qr, pos, Kg[z], Vg[z], dOg[z, r0:r0 + chunk], causal, scale)
            Pk, dSk = P[:, keys], dS[:, keys]                     # [rows, n]
            Q2, dO2 = Qr * Qr, dOg[z, r0:r0 + chunk] ** 2
            vk += (dSk * dSk).T @ Q2
            vq += (Pk * Pk * sd2[:, None]).T @ Q2
            vv += (Pk * Pk).T @ dO2
            cnt += (Pk > 0).sum(0)
        sig_k = abs(scale) * torch.sqrt((U * U / 3) * vk + vq)
        sig_v = torch.sqrt((U * U / 3) * vv)
        acc = torch.tensor([_acc(int(c)) for c in cnt.tolist()], dtype=torch.float64,
                           device=device)[:, None]
        res[0][sel] = sig_k.cpu().numpy()
        res[1][sel] = (acc * abs(scale) * torch.sqrt(vk)).cpu().numpy()
        res[2][sel] = sig_v.cpu().numpy()
        res[3][sel] = (acc * torch.sqrt(vv)).cpu().numpy()
    return tuple(res)


def check(name: str, got, ref, sigma, acc) -> dict:
    """Asserts every element within K_SIGMA sigma + acc + u |ref| of the
    oracle, and the RMS of the errors in units of the model's standard
    deviation (sigma together with the output rounding, u |ref| / sqrt(3))
    within 1.5: sigma bounds each rounding's deviation from above, so a
    kernel that follows the model stays near or below 1 on average.  Returns
    the statistics (printed too)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    sigma = np.asarray(sigma, np.float64).reshape(ref.shape)
    acc = np.asarray(acc, np.float64).reshape(ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = np.abs(got - ref)
    allow = K_SIGMA * sigma + acc + U * np.abs(ref) + 1e-30
    ratio = err / allow
    live = sigma > 0
    sd = np.sqrt(sigma * sigma + (U * ref) ** 2 / 3)
    z = err[live] / sd[live]
    st = {
        "rel_fro": float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)),
        "max_err_over_max_ref": float(err.max() / max(np.abs(ref).max(), 1e-30)),
        "max_err_over_allowance": float(ratio.max()),
        "max_z": float(z.max()) if z.size else 0.0,
        "rms_z": float(np.sqrt(np.mean(z * z))) if z.size else 0.0,
        "n": int(err.size),
    }
    print(f"{name}: {st}")
    assert ratio.max() <= 1.0, f"{name}: an element beyond its allowance: {st}"
    # elements with sigma = 0 (no visible term) must be exact up to rounding
    assert (err[~live] <= U * np.abs(ref[~live]) + 1e-30).all(), f"{name}: {st}"
    assert st["rms_z"] <= 1.5, f"{name}: errors larger than the rounding model: {st}"
    return st
