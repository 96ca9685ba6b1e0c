"""Move the seeded host inputs to a CUDA device and allocate result buffers.

Plumbing for the tests and the bench (torch tensors for device memory); no
arithmetic of the verify step happens here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import NINE_B, RMS_EPS, ROPE_THETA, TINY, Batch, Weights  # noqa: F401


def _t(a: np.ndarray, dev, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(dev, non_blocking=False)


def config(dims: dict, gamma_max: int, fmt: str = "bf16") -> dict:
    return dict(hidden=dims["hidden"], n_q=dims["n_q"], n_kv=dims["n_kv"], head_dim=dims["head_dim"],
                ffn=dims["ffn"], vocab=dims["vocab"], page_size=dims["page"], gamma_max=gamma_max,
                weight_format=0 if fmt == "bf16" else 1, rms_eps=RMS_EPS, rope_theta=ROPE_THETA)


def weights_to_device(W: Weights, dev="cuda") -> dict:
    bf = torch.bfloat16
    d = dict(emb=_t(W.emb.view(np.int16), dev, bf), w_lm=_t(W.w_lm.view(np.int16), dev, bf),
             g_attn=_t(W.g_attn.view(np.int16), dev, bf), g_ffn=_t(W.g_ffn.view(np.int16), dev, bf),
             g_final=_t(W.g_final.view(np.int16), dev, bf))
    for name in ("qkv", "o", "gate", "up", "down"):
        w = W.proj[name]
        if isinstance(w, tuple):
            d["w_" + name] = _t(w[0], dev)
            d["s_" + name] = _t(w[1].view(np.int16), dev, torch.float16)
        else:
            d["w_" + name] = _t(w.view(np.int16), dev, bf)
    return d


def batch_to_device(b: Batch, dev="cuda") -> dict:
    i32 = np.int32
    d = dict(B=b.B, R=b.R, G=b.G,
             seq_lens=_t(b.seq_lens.astype(i32), dev), draft_lens=_t(b.draft_lens.astype(i32), dev),
             tokens=_t(b.tokens.astype(i32), dev),
             draft_probs=_t(b.draft_probs.astype(np.float32).reshape(b.G, b.dims["vocab"]), dev),
             uniforms=_t(b.uniforms.astype(np.float32), dev),
             kv_pool=_t(b.kv_pool.view(np.int16), dev, torch.bfloat16),
             num_pool_pages=int(b.kv_pool.shape[0]),
             page_table=_t(b.page_table.astype(i32), dev), num_pages=_t(b.num_pages.astype(i32), dev),
             free_pages=_t(b.free_pages.astype(i32), dev),
             num_free_in=_t(np.array([b.num_free], i32), dev))
    d["num_free_out"] = d["num_free_in"]
    if b.gen_counts is not None:
        d["gen_counts"] = _t(b.gen_counts.astype(i32), dev)
    if b.gen_limits is not None:
        d["gen_limits"] = _t(b.gen_limits.astype(i32), dev)
    return d


def alloc_result(B: int, R: int, V: int, gamma_max: int, max_pages: int, dev="cuda",
                 logits: bool = False, probs: bool = False, next_view: bool = True) -> dict:
    z = lambda n: torch.zeros(n, dtype=torch.int32, device=dev)  # noqa: E731
    r = dict(accepted=z(B), final_tokens=z(B), emitted_tokens=z(R), emitted_offsets=z(B + 1),
             new_seq_lens=z(B), finished=z(B), new_gen_counts=z(B),
             accept_tested=z(max(gamma_max, 1)), accept_accepted=z(max(gamma_max, 1)), status=z(1))
    if next_view:
        r.update(next_src=z(B), num_live=z(1), next_seq_lens=z(B), next_num_pages=z(B),
                 next_page_table=torch.full((B, max_pages), -1, dtype=torch.int32, device=dev),
                 next_gen_counts=z(B))
    if logits:
        r["logits"] = torch.zeros((R, V), dtype=torch.float32, device=dev)
    if probs:
        r["probs"] = torch.zeros((R, V), dtype=torch.float32, device=dev)
    return r


# ---------------------------------------------------------------------------
# inputs drawn on the device (full-size runs whose KV pool and draft
# distributions are too large to draw on the host every step)
# ---------------------------------------------------------------------------

def _generator(key: int):
    g = torch.Generator(device="cuda")
    g.manual_seed(key & ((1 << 63) - 1))
    return g


def normal_bf16_device_(t: torch.Tensor, key: int) -> torch.Tensor:
    """Fill a bf16 device tensor with N(0, 1) draws from a seeded device generator."""
    return t.normal_(generator=_generator(key))


def draft_probs_device(G: int, V: int, key: int, sigma: float = 2.0) -> torch.Tensor:
    """q = softmax(N(0, sigma^2) logits) per draft row, fp32 [G, V], drawn on the device."""
    if G == 0:
        return torch.zeros((0, V), dtype=torch.float32, device="cuda")
    z = torch.randn((G, V), generator=_generator(key), device="cuda", dtype=torch.float32)
    return torch.softmax(z * sigma, dim=1)


def retarget_draft_probs_device(q: torch.Tensor, probs: torch.Tensor, tokens: torch.Tensor, gamma: int,
                                alphas: torch.Tensor) -> None:
    """Device form of the input recipe of ``retarget_draft_probs`` for a batch in
    which every slot drafts ``gamma`` tokens: q_i(x_{i+1}) = p_i(x_{i+1}) / alpha_b,
    the rest of q_i rescaled to sum to one, so every draft is accepted with
    probability alpha_b.  q [B*gamma, V] is rewritten in place; probs [B*(gamma+1), V]
    are the target's probabilities from a prepass; alphas [B] float64."""
    if gamma == 0 or q.shape[0] == 0:
        return
    B = alphas.shape[0]
    b = torch.arange(B, device=q.device).repeat_interleave(gamma)
    i = torch.arange(gamma, device=q.device).repeat(B)
    r = b * (gamma + 1) + i
    x = tokens[r + 1].long()
    g = torch.arange(B * gamma, device=q.device)
    target = probs[r, x].double() / alphas.to(q.device)[b]
    qx = q[g, x].double()
    scale = ((1.0 - target) / (1.0 - qx)).float()
    q.mul_(scale[:, None])
    q[g, x] = target.float()
