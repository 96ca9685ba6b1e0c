"""Shared pieces of the GPU parity tests: running the CUDA path on seeded
inputs and comparing it with the oracle under the tolerances the tests state.
"""
from __future__ import annotations

import numpy as np

from oracle import verify_step as o
import workloads as wl

# tolerances stated for the bf16 forward (bf16 weights and KV cache)
LOGIT_TOL_REL_RMS = 1e-2      # max |dlogit| <= 1e-2 * rms(logits)
PROB_TOL_ABS = 1e-3           # max |dp| <= 1e-3
# derived: |dz| <= 1e-2 rms with rms <= 1.3 moves p by at most exp(2 * 1.3e-2) - 1 < 3 %
PROB_TOL_REL = 3e-2
# an acceptance decision or a sampled token is only required to agree when
# the oracle's margin exceeds what that probability error can move
DECISION_REL = 3e-2


def engine_for(dims, gamma_max, W_dev, max_rows, max_slots, fmt="bf16"):
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine
    from workloads import device as wd
    return VerifyEngine(wd.config(dims, gamma_max, fmt), W_dev, max_rows, max_slots)


def run_step(eng, batch: wl.Batch, logits=True, probs=True):
    import torch
    from workloads import device as wd
    bd = wd.batch_to_device(batch)
    res = wd.alloc_result(batch.B, batch.R, batch.dims["vocab"], batch.gamma_max, batch.page_table.shape[1],
                          logits=logits, probs=probs)
    eng.verify_step(bd, res)
    status = eng.read_status(res["status"])
    torch.cuda.synchronize()
    return status, to_numpy(res), to_numpy(bd)


def to_numpy(d: dict) -> dict:
    import torch
    out = {}
    for k, v in d.items():
        if hasattr(v, "cpu"):
            if v.dtype == torch.bfloat16:
                out[k] = v.view(torch.int16).cpu().numpy().view(np.uint16)
            else:
                out[k] = v.cpu().numpy()
        else:
            out[k] = v
    return out


def compare_logits(z_gpu, z_or, p_gpu=None, p_or=None):
    rms = float(np.sqrt(np.mean(z_or ** 2)))
    dz = float(np.max(np.abs(z_gpu.astype(np.float64) - z_or)))
    assert dz <= LOGIT_TOL_REL_RMS * rms, f"logits: max|d| {dz:.3e} > {LOGIT_TOL_REL_RMS} * rms {rms:.3e}"
    if p_gpu is not None:
        dp = np.abs(p_gpu.astype(np.float64) - p_or)
        assert float(dp.max()) <= PROB_TOL_ABS, f"probs: max|d| {dp.max():.3e}"
        big = p_or > 1e-7
        rel = float((dp[big] / p_or[big]).max())
        assert rel <= PROB_TOL_REL, f"probs: max rel {rel:.3e}"
    return dz / rms


def _ambiguous(p, q, u, rel=DECISION_REL):
    if p <= 0:
        return False
    return abs(float(np.float32(u) * np.float32(q)) - p) <= rel * p or abs(p - q) <= rel * p


def check_acceptance(batch: wl.Batch, p_or: np.ndarray, acc_gpu, fin_gpu):
    """Acceptance counts and final tokens against the oracle, up to decision margins.

    Returns the number of slots whose result had to be judged by margin.
    """
    p32 = p_or.astype(np.float32)
    roff = wl.row_offsets(batch.draft_lens)
    goff = np.concatenate([[0], np.cumsum(batch.draft_lens)])
    judged = 0
    for b in range(batch.B):
        g = int(batch.draft_lens[b])
        r0 = int(roff[b])
        drafts = batch.tokens[r0 + 1: r0 + 1 + g]
        q = batch.draft_probs[int(goff[b]): int(goff[b]) + g]
        u = batch.uniforms[r0: r0 + g + 1]
        a_or, t_or = o.accept_and_sample(p32[r0: r0 + g + 1], q, drafts, u)
        amb = None
        for i in range(g):
            x = int(drafts[i])
            if _ambiguous(float(p32[r0 + i, x]), float(q[i, x]), float(u[i])):
                amb = i
                break
            if not o.accepts(p32[r0 + i, x], q[i, x], u[i]):
                break
        a_g = int(acc_gpu[b])
        if amb is None or amb > a_or:
            assert a_g == a_or, f"slot {b}: accepted {a_g} vs oracle {a_or}"
        else:
            judged += 1
            assert a_g >= amb, f"slot {b}: accepted {a_g} before the ambiguous draft {amb}"
            continue
        t_g = int(fin_gpu[b])
        if t_g == t_or:
            continue
        # the GPU's token must sit at the oracle's CDF point within the probability tolerance
        if a_or < g:
            w = np.maximum(np.float32(0), p32[r0 + a_or] - q[a_or])
            if not np.any(np.floor(w.astype(np.float64) * 2.0 ** 32) > 0):
                w = p32[r0 + a_or]
        else:
            w = p32[r0 + g]
        W = np.floor(w.astype(np.float64) * 2.0 ** 32)
        cum = np.cumsum(W)
        S = cum[-1]
        T = np.floor(S * np.floor(float(u[g]) * 2 ** 24) / 2 ** 24)
        lo = cum[t_g - 1] if t_g > 0 else 0.0
        judged += 1
        assert lo - DECISION_REL * S <= T <= cum[t_g] + DECISION_REL * S, (
            f"slot {b}: token {t_g} vs oracle {t_or} outside the tolerance of the CDF")
    return judged
