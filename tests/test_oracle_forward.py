"""Pins for the oracle's forward pass (CPU only).

The oracle is checked against library routines (torch's bf16 conversion,
rms_norm, silu, scaled_dot_product_attention with GQA, softmax), an
independent complex-number formulation of rotary embedding, hand-computed
int4 codes, and invariants the method must satisfy: causality inside the
draft block, independence from where pages sit in the pool, and batch
equivalence (a sequence's rows are the same alone or in a ragged batch; the
"output equivalence" the Compute Slack post's section "The batch also goes
ragged" demands of batched speculation).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import verify_step as o
import workloads as wl


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_round_bf16_matches_torch():
    g = np.random.default_rng(0)
    x32 = (g.standard_normal(200000) * np.exp(g.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.round_bf16(x32.astype(np.float64)), ref)
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert o.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert o.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    assert o.round_bf16(np.array([-(1 + 2 ** -8 + 2 ** -30)]))[0] == -(1 + 2 ** -7)


def test_round_bf16_other_is_the_far_neighbour():
    """The other rounding of x is the adjacent bf16 value on x's far side."""
    g = np.random.default_rng(5)
    x32 = (g.standard_normal(50000) * np.exp(g.uniform(-10, 10, 50000))).astype(np.float32)
    x = x32.astype(np.float64)
    near = o.round_bf16(x)
    far = o.round_bf16_other(x, near)
    t = torch.from_numpy(near.astype(np.float32)).to(torch.bfloat16)
    up = torch.nextafter(t, torch.full_like(t, float("inf"))).double().numpy()
    down = torch.nextafter(t, torch.full_like(t, float("-inf"))).double().numpy()
    exact = x == near
    assert np.array_equal(far[exact], near[exact])
    m = ~exact
    assert np.array_equal(far[m], np.where(x[m] > near[m], up[m], down[m]))
    # across a power of two the spacing changes: 1 - 2^-10 rounds to 1, its far neighbour is 1 - 2^-8
    assert o.round_bf16_other(np.array([1 - 2 ** -10]), np.array([1.0]))[0] == 1 - 2 ** -8
    assert o.round_bf16_other(np.array([1 + 2 ** -9]), np.array([1.0]))[0] == 1 + 2 ** -7


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]          # skip inf/nan
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.bf16_to_f64(bits), ref)


def test_int4_dequant_hand_cases():
    # byte 0x8F: low nibble 0xF = -1 (even k), high nibble 0x8 = -8 (odd k)
    # byte 0x70: low 0 , high 7
    packed = np.zeros((1, 16), dtype=np.uint8)
    packed[0, 0] = 0x8F
    packed[0, 1] = 0x70
    packed[0, 15] = 0x21
    scales = np.array([[np.float16(0.5).view(np.uint16)]], dtype=np.uint16)
    w = o.dequant_int4_g32(packed, scales)
    assert w.shape == (1, 32)
    assert list(w[0, :4]) == [-0.5, -4.0, 0.0, 3.5]
    assert list(w[0, 30:]) == [0.5, 1.0]
    # second group uses the second scale
    packed2 = np.full((1, 32), 0x11, dtype=np.uint8)
    sc2 = np.array([[np.float16(1.0).view(np.uint16), np.float16(0.25).view(np.uint16)]], dtype=np.uint16)
    w2 = o.dequant_int4_g32(packed2, sc2)
    assert np.all(w2[0, :32] == 1.0) and np.all(w2[0, 32:] == 0.25)


# ---------------------------------------------------------------------------
# rotary embedding: complex-number formulation and its invariants
# ---------------------------------------------------------------------------

def _rope_complex(x, pos, theta):
    d = x.shape[-1]
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = np.array([theta ** (-2.0 * j / d) for j in range(half)])
    rot = np.exp(1j * pos[:, None, None] * freq[None, None, :])
    w = z * rot
    return np.concatenate([w.real, w.imag], axis=-1)


def test_rope_matches_complex_rotation():
    g = np.random.default_rng(1)
    x = g.standard_normal((5, 3, 64))
    pos = np.array([0, 1, 17, 2048, 16000])
    assert np.allclose(o.rope(x, pos, 1e6), _rope_complex(x, pos, 1e6), atol=1e-12)
    # position 0 is the identity
    assert np.array_equal(o.rope(x[:1], np.array([0]), 1e6), x[:1])


def test_rope_scores_depend_on_relative_position_only():
    g = np.random.default_rng(2)
    q = g.standard_normal((1, 1, 128))
    k = g.standard_normal((1, 1, 128))
    s1 = (o.rope(q, np.array([100]), 1e6) * o.rope(k, np.array([40]), 1e6)).sum()
    s2 = (o.rope(q, np.array([1060]), 1e6) * o.rope(k, np.array([1000]), 1e6)).sum()
    assert s1 == pytest.approx(s2, rel=1e-9, abs=1e-9)


# ---------------------------------------------------------------------------
# the forward against torch library routines (float64)
# ---------------------------------------------------------------------------

def _bf(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64)


def _w(bits):
    return torch.from_numpy(o.bf16_to_f64(bits))


def _torch_forward(dims, W, batch, eps=1e-6, theta=1e6, drop_gain=False, gqa_tile=False):
    """Same layer through torch.nn.functional, bf16 rounding at the same points."""
    nq, nkv, d, P = dims["n_q"], dims["n_kv"], dims["head_dim"], dims["page"]
    H = dims["hidden"]
    offs = wl.row_offsets(batch.draft_lens)
    pool = o.bf16_to_f64(batch.kv_pool)
    x0 = _w(W.emb[batch.tokens])
    g_attn = None if drop_gain else _w(W.g_attn)
    h1 = F.rms_norm(x0, (H,), g_attn, eps)
    qkv = F.linear(h1, _w(W.proj["qkv"]))
    R = qkv.shape[0]
    pos = np.concatenate([np.arange(batch.seq_lens[b], batch.seq_lens[b] + batch.draft_lens[b] + 1)
                          for b in range(batch.B)])
    q = qkv[:, : nq * d].reshape(R, nq, d).numpy()
    k = qkv[:, nq * d:(nq + nkv) * d].reshape(R, nkv, d).numpy()
    v = qkv[:, (nq + nkv) * d:].reshape(R, nkv, d)
    q = torch.from_numpy(_rope_complex(q, pos, theta))
    k = _bf(_rope_complex(k, pos, theta))
    v = _bf(v.numpy())
    outs = []
    for b in range(batch.B):
        L, gm = int(batch.seq_lens[b]), int(batch.draft_lens[b])
        r0 = int(offs[b])
        n = L + gm + 1
        Kc = torch.zeros(nkv, n, d, dtype=torch.float64)
        Vc = torch.zeros(nkv, n, d, dtype=torch.float64)
        for t in range(L):
            pg = batch.page_table[b, t // P]
            Kc[:, t] = torch.from_numpy(pool[pg, :, 0, t % P])
            Vc[:, t] = torch.from_numpy(pool[pg, :, 1, t % P])
        Kc[:, L:] = k[r0:r0 + gm + 1].transpose(0, 1)
        Vc[:, L:] = v[r0:r0 + gm + 1].transpose(0, 1)
        qb = q[r0:r0 + gm + 1].transpose(0, 1)                       # [nq, rows, d]
        mask = torch.zeros(gm + 1, n, dtype=torch.bool)
        for i in range(gm + 1):
            mask[i, : L + i + 1] = True
        if gqa_tile:
            Kg, Vg = Kc.repeat(nq // nkv, 1, 1), Vc.repeat(nq // nkv, 1, 1)
        else:
            Kg, Vg = Kc.repeat_interleave(nq // nkv, 0), Vc.repeat_interleave(nq // nkv, 0)
        ob = F.scaled_dot_product_attention(qb[None], Kg[None], Vg[None], attn_mask=mask)[0]
        outs.append(ob.transpose(0, 1).reshape(gm + 1, nq * d))
    att = torch.cat(outs)
    x1 = x0 + F.linear(att, _w(W.proj["o"]))
    h2 = F.rms_norm(x1, (H,), _w(W.g_ffn), eps)
    act = F.silu(F.linear(h2, _w(W.proj["gate"]))) * F.linear(h2, _w(W.proj["up"]))
    x2 = x1 + F.linear(act, _w(W.proj["down"]))
    h3 = _bf(F.rms_norm(x2, (H,), _w(W.g_final), eps).numpy())
    z = F.linear(h3, _w(W.w_lm))
    return z.numpy(), torch.softmax(z, dim=-1).numpy()


@pytest.fixture(scope="module")
def tiny():
    W = wl.make_weights(wl.TINY, 1)
    # a sequence with an empty cache next to a ragged one
    batch = wl.make_batch(wl.TINY, 1, seq_lens=[0, 37, 128], draft_lens=[2, 0, 3], gamma_max=3,
                          extra_pages=4)
    return W, batch


def test_forward_matches_torch_library(tiny):
    W, batch = tiny
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                   batch.draft_lens, batch.tokens)
    z_ref, p_ref = _torch_forward(batch.dims, W, batch)
    rms = np.sqrt(np.mean(z_ref ** 2))
    assert np.max(np.abs(fw["logits"] - z_ref)) < 1e-6 * rms
    assert np.max(np.abs(fw["probs"] - p_ref)) < 1e-7


@pytest.mark.parametrize("mistake", ["drop_gain", "gqa_tile"])
def test_forward_pin_has_power(tiny, mistake):
    """A planted mistake in the reference differs from the oracle by far more than the pin allows."""
    W, batch = tiny
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                   batch.draft_lens, batch.tokens)
    z_bad, _ = _torch_forward(batch.dims, W, batch, **{mistake: True})
    rms = np.sqrt(np.mean(z_bad ** 2))
    assert np.max(np.abs(fw["logits"] - z_bad)) > 1e-2 * rms


def test_kv_written_at_row_positions(tiny):
    """Row i of a sequence writes K/V at position L + i; at L = 0 row 0's K is unrotated."""
    W, batch = tiny
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                   batch.draft_lens, batch.tokens)
    keys = sorted(fw["kv_rows"].keys())
    expect = sorted((b, int(batch.seq_lens[b]) + i) for b in range(batch.B)
                    for i in range(int(batch.draft_lens[b]) + 1))
    assert keys == expect
    d, nq, nkv = 64, 4, 2
    h1 = torch.from_numpy(fw["h1"][0:1])
    k_raw = F.linear(h1, _w(W.proj["qkv"]))[0, nq * d:(nq + nkv) * d].reshape(nkv, d)
    assert np.allclose(fw["kv_rows"][(0, 0)][0], _bf(k_raw.numpy()).numpy(), rtol=2 ** -8, atol=0)


def test_forward_flips_take_the_other_rounding(tiny):
    """A flipped K/V element holds the far bf16 neighbour of its exact value; a flipped
    h3 element moves the logits by exactly (its change) x (its LM-head column)."""
    W, batch = tiny
    args = (batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens, batch.tokens)
    fw = o.forward(*args)
    same = o.forward(*args, flips=set())
    assert np.array_equal(fw["logits"], same["logits"])
    r = int(wl.row_offsets(batch.draft_lens)[2]) + 1          # slot 2, draft row 1
    pos = int(batch.seq_lens[2]) + 1
    fk = o.forward(*args, flips={("k", r, 1, 5), ("v", r, 0, 7)})
    k0, v0 = fw["kv_rows"][(2, pos)]
    k1, v1 = fk["kv_rows"][(2, pos)]
    assert np.count_nonzero(k0 != k1) == 1 and np.count_nonzero(v0 != v1) == 1
    assert k1[1, 5] == o.round_bf16_other(fw["k_pre"][r, 1, 5], k0[1, 5])
    assert v1[0, 7] == o.round_bf16_other(fw["v_pre"][r, 0, 7], v0[0, 7])
    # rows before the flipped one in its sequence, and other sequences, are unchanged
    assert np.array_equal(fk["logits"][:r], fw["logits"][:r])
    assert not np.array_equal(fk["logits"][r], fw["logits"][r])
    fh = o.forward(*args, flips={("h3", r, 11)})
    dh = fh["h3"][r, 11] - fw["h3"][r, 11]
    assert dh != 0 and np.array_equal(np.delete(fh["h3"][r], 11), np.delete(fw["h3"][r], 11))
    col = o.bf16_to_f64(W.w_lm[:, 11])
    assert np.allclose(fh["logits"][r] - fw["logits"][r], dh * col, rtol=1e-9, atol=1e-12)


def test_causal_inside_draft_block(tiny):
    """Changing draft token i changes no row before i."""
    W, batch = tiny
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                   batch.draft_lens, batch.tokens)
    tok2 = batch.tokens.copy()
    r_last = int(wl.row_offsets(batch.draft_lens)[3]) - 1    # last row of slot 2
    tok2[r_last] = (tok2[r_last] + 1) % batch.dims["vocab"]
    fw2 = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                    batch.draft_lens, tok2)
    assert np.array_equal(fw["logits"][:r_last], fw2["logits"][:r_last])
    assert not np.array_equal(fw["logits"][r_last], fw2["logits"][r_last])


def test_page_placement_does_not_matter(tiny):
    W, batch = tiny
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                   batch.draft_lens, batch.tokens)
    g = np.random.default_rng(3)
    n = batch.kv_pool.shape[0]
    perm = g.permutation(n)                      # new page j holds old page perm[j]
    inv = np.argsort(perm)
    pool2 = batch.kv_pool[perm]
    pt2 = np.where(batch.page_table >= 0, inv[np.maximum(batch.page_table, 0)], -1)
    fw2 = o.forward(batch.dims, W, pool2, pt2, batch.seq_lens, batch.draft_lens, batch.tokens)
    assert np.array_equal(fw["logits"], fw2["logits"])


def test_batch_equivalence(tiny):
    """Each sequence's rows are identical alone and inside the ragged batch."""
    W, batch = tiny
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                   batch.draft_lens, batch.tokens)
    offs = wl.row_offsets(batch.draft_lens)
    for b in range(batch.B):
        one = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                        batch.draft_lens, batch.tokens, slots=[b])
        assert np.array_equal(one["logits"], fw["logits"][offs[b]:offs[b + 1]])


def test_attention_single_key_returns_value():
    g = np.random.default_rng(4)
    q = g.standard_normal(16)
    K = g.standard_normal((1, 16))
    V = g.standard_normal((1, 16))
    assert np.allclose(o.attention_one(q, K, V), V[0])
    # equal keys: uniform weights, mean of values
    K = np.repeat(K, 5, axis=0)
    V = g.standard_normal((5, 16))
    assert np.allclose(o.attention_one(q, K, V), V.mean(axis=0))


def test_int4_forward_uses_dequantized_weights():
    """The int4 layer equals the bf16-free float64 layer built from s * code."""
    W = wl.make_weights(wl.TINY, 1, fmt="int4")
    batch = wl.make_batch(wl.TINY, 1, seq_lens=[20], draft_lens=[1], gamma_max=1)
    x = np.random.default_rng(5).standard_normal((3, 256))
    packed, scales = W.proj["gate"]
    y = o.linear(x, W.proj["gate"])
    codes = np.zeros((packed.shape[0], packed.shape[1] * 2))
    for n in range(packed.shape[0]):
        for k in range(packed.shape[1] * 2):
            byte = int(packed[n, k // 2])
            nib = (byte >> (4 * (k % 2))) & 0xF
            codes[n, k] = nib - 16 if nib >= 8 else nib
    s = np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=1)
    assert np.allclose(y, x @ (codes * s).T, rtol=1e-12, atol=1e-12)
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens,
                   batch.draft_lens, batch.tokens)
    assert np.all(np.isfinite(fw["logits"]))
