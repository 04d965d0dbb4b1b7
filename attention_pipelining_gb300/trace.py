"""Summaries of the kernel timeline recorded by ``attn_fwd_trace``.

For each traced CTA the stamps give, per KV block j, when each warp role
passed its hand-off points.  ``summarize`` turns them into the per-iteration
numbers that show where a pipelined schedule loses time: how long each
softmax pass takes, how long the tensor-core issuer waits after P is ready,
and the steady-state period of one KV block.
"""
from __future__ import annotations

import numpy as np

from . import TRACE_EVENTS

EV = {name: i for i, name in enumerate(TRACE_EVENTS)}


def _med(x):
    x = np.asarray(x, dtype=np.float64)
    x = x[np.isfinite(x)]
    return float(np.median(x)) if x.size else float("nan")


def summarize(trace, n_blocks: int) -> dict:
    """trace: int64 array [ctas, 16, blocks] (SM clock cycles).  Medians over CTAs and over
    the steady-state blocks (the first and last two are left out)."""
    t = np.asarray(trace, dtype=np.float64)
    t[t == 0] = np.nan
    n = min(n_blocks, t.shape[2])
    js = np.arange(2, max(3, n - 2))

    def ev(name):
        return t[:, EV[name], :n]

    out = {}
    for s in ("0", "1"):
        wake, loaded, done = ev(f"sm{s}_wake"), ev(f"sm{s}_loaded"), ev(f"sm{s}_done")
        out[f"softmax{s}_cyc"] = _med((done - wake)[:, js])
        out[f"softmax{s}_tmem_load_cyc"] = _med((loaded - wake)[:, js])
        out[f"softmax{s}_compute_cyc"] = _med((done - loaded)[:, js])
        out[f"pv{s}_issue_after_p_cyc"] = _med((ev(f"mma_pv{s}") - done)[:, js])
        # S_t(j+1) issued -> softmax t wakes on it
        s_issue = ev(f"mma_s{s}")
        out[f"s{s}_issue_to_wake_cyc"] = _med((wake[:, js] - s_issue[:, js]))
        out[f"period{s}_cyc"] = _med(np.diff(wake, axis=1)[:, js[:-1]])
    out["corr0_after_sm0_done_cyc"] = _med((ev("corr0") - ev("sm0_done"))[:, js])
    out["load_k_lead_cyc"] = _med((ev("mma_s0") - ev("load_k"))[:, js])
    end = t[:, EV["end"], 0]
    start = np.nanmin(t[:, :, 0], axis=1)
    out["cta_cyc"] = _med(end - start)
    out["blocks"] = n
    return out
