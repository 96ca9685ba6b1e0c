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


# ---------------------------------------------------------------------------
# roundings that either side may take
# ---------------------------------------------------------------------------
# K, V and the LM-head input are rounded to bf16 from values the GPU carries
# with an absolute error of about 2^-18 times the rms of the vector they
# belong to (one K/V head, or the row of h3): fp32 activations enter the
# tensor cores as bf16 hi + lo (16 significant bits) and fp32 accumulation
# adds less; the largest disagreement seen on the 9B-class layer is 2^-17.
# Any bf16 value that rounds from a point within TIE_WINDOW * rms of the exact
# value is a valid result: the nearest one, its other neighbour when the
# exact value sits near a tie, and, for elements much smaller than the rms,
# values a few spacings away.  The window is 8x the largest seen error.
TIE_WINDOW = 2.0 ** -14
MAX_CANDIDATES = 12


def _tie_distance(pre, axis):
    near = o.round_bf16(pre)
    far = o.round_bf16_other(pre, near)
    scale = np.sqrt(np.mean(pre ** 2, axis=axis, keepdims=True))
    d = np.abs(pre - 0.5 * (near + far)) / np.maximum(scale, 1e-300)
    return np.where(near == pre, np.inf, d), near, far


def check_kv_written(batch, fw, pool, pt_before):
    """Each verified row's K/V sits in its page at position L + i and is a bf16
    rounding of a point within TIE_WINDOW * rms of the oracle's exact value.
    Returns the number of elements that differ from the nearest rounding."""
    page = batch.dims["page"]
    offs = wl.row_offsets(batch.draft_lens)
    local = {int(r): n for n, r in enumerate(fw["rows"])}
    other = 0
    for (b, pos) in fw["kv_rows"]:
        n = local[int(offs[b]) + pos - int(batch.seq_lens[b])]
        pg = pt_before[b, pos // page]
        for kind, kv in (("k", 0), ("v", 1)):
            got = o.bf16_to_f64(pool[pg, :, kv, pos % page, :])
            pre = fw[kind + "_pre"][n]
            e = TIE_WINDOW * np.sqrt(np.mean(pre ** 2, axis=1, keepdims=True))
            ok = (o.round_bf16(pre - e) <= got) & (got <= o.round_bf16(pre + e))
            assert ok.all(), (kind, b, pos, np.argwhere(~ok)[:4])
            other += int(np.count_nonzero(got != o.round_bf16(pre)))
    return other


def _row_errors(z_gpu, p_gpu, z_or, p_or, tol):
    dz = np.max(np.abs(z_gpu.astype(np.float64) - z_or), axis=-1)
    bad = dz > tol
    if p_gpu is not None:
        dp = np.abs(p_gpu.astype(np.float64) - p_or)
        rel = np.where(p_or > 1e-7, dp / np.maximum(p_or, 1e-300), 0.0)
        bad |= (dp.max(-1) > PROB_TOL_ABS) | (rel.max(-1) > PROB_TOL_REL)
    return dz, bad


def compare_step(batch, W, fw, z_gpu, p_gpu=None):
    """Logits within LOGIT_TOL_REL_RMS * rms and probabilities within PROB_TOL_ABS
    (and PROB_TOL_REL) of the oracle.  A sequence with a row outside must match,
    within the same tolerances, the oracle's result under some choice of the
    other rounding for K/V/h3 values inside the tie window (its rows up to the
    failing one, the nearest MAX_CANDIDATES ties): a result that is just as
    valid.  Returns (probs the acceptance check should use, {slot: flips}).
    """
    z_or, p_or = fw["logits"], fw["probs"]
    rms = float(np.sqrt(np.mean(z_or ** 2)))
    tol = LOGIT_TOL_REL_RMS * rms
    dz, bad = _row_errors(z_gpu, p_gpu, z_or, p_or, tol)
    p_valid = p_or.copy()
    explained = {}
    if not bad.any():
        return p_valid, explained
    offs = wl.row_offsets(batch.draft_lens)
    row_slot = np.repeat(np.arange(batch.B), np.asarray(batch.draft_lens) + 1)
    slots = sorted(set(int(row_slot[r]) for r in np.nonzero(bad)[0]))
    assert len(slots) <= max(2, batch.B // 4), f"{len(slots)} sequences outside tolerance: {dz.max() / rms:.3e} rms"
    args = (batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens, batch.tokens)
    for b in slots:
        r0, r1 = int(offs[b]), int(offs[b + 1])
        bad_rows = [r for r in range(r0, r1) if bad[r]]
        last = max(bad_rows)
        cands = []
        for r in range(r0, last + 1):
            for kind in ("k", "v"):
                d = _tie_distance(fw[kind + "_pre"][r], axis=1)[0]
                for h, j in np.argwhere(d <= TIE_WINDOW):
                    cands.append((float(d[h, j]), (kind, r, int(h), int(j))))
        for r in bad_rows:
            d = _tie_distance(fw["h3_pre"][r], axis=0)[0]
            for j in np.nonzero(d <= TIE_WINDOW)[0]:
                cands.append((float(d[j]), ("h3", r, int(j))))
        cands = [c for _, c in sorted(cands)[:MAX_CANDIDATES]]
        assert cands, f"slot {b}: rows {bad_rows} outside tolerance ({dz[bad_rows].max() / rms:.3e} rms), no tie in reach"
        sel = [r - r0 for r in bad_rows]
        err = (z_gpu[bad_rows].astype(np.float64) - z_or[bad_rows]).ravel()
        eff = np.stack([(o.forward(*args, slots=[b], flips={c})["logits"][sel] - z_or[bad_rows]).ravel()
                        for c in cands])
        # fewest flips first: the first choice that leaves the rows well inside the
        # tolerance (half of it, before the exact re-run), else the closest one
        best, best_res = None, np.inf
        for mask in sorted(range(1, 1 << len(cands)), key=lambda m: (bin(m).count("1"), m)):
            pick = [i for i in range(len(cands)) if mask >> i & 1]
            res = float(np.max(np.abs(err - eff[pick].sum(0))))
            if res < best_res:
                best, best_res = pick, res
            if res <= 0.5 * tol:
                break
        flips = {cands[i] for i in best}
        alt = o.forward(*args, slots=[b], flips=flips)
        _, still = _row_errors(z_gpu[r0:r1], None if p_gpu is None else p_gpu[r0:r1], alt["logits"],
                               alt["probs"], tol)
        assert not still.any(), (f"slot {b}: rows {bad_rows} outside tolerance ({dz[bad_rows].max() / rms:.3e} rms) "
                                 f"under every tie choice tried")
        p_valid[r0:r1] = alt["probs"]
        explained[b] = sorted(flips)
    return p_valid, explained


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
