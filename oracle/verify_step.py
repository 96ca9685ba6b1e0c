"""CPU oracle for the ragged batched speculative-verify step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product
(the CUDA library and its Python binding) never calls it, and it shares no
code with the product: it imports numpy and the seeded input generator only.

Plain, slow and direct: numpy in float64, one step after another in the order
the method states them, no blocking or fusion beyond chunking the rows of a
weight matrix to bound host memory (each output is still one dot product).

What it computes, and where the pages say so:

* One verify pass over the gamma_b + 1 rows of every live sequence, reading
  the weights once ("Speculative Decoding at High Batch Size", section "Why
  do the headline speedups all come from batch 1?"; the splicedso primer,
  section "The idea": the large model checks all guesses in one pass).
* Acceptance of a prefix of the drafts plus one token of the target's own
  (primer, "The idea"; "Speculative Decoding and Batching Compete for the Same
  Compute Slack on RDNA4", section "The batch also goes ragged"), by
  rejection sampling so that the output distribution is unchanged ("High
  Batch Size" post, FAQ "Does speculative decoding change the output of the
  model?", citing Leviathan, Kalman and Matias).
* Realignment of each sequence's KV length, next position and page list from
  its own accepted count, with no padding to the longest run ("Compute Slack"
  post, section "The batch also goes ragged"), and stable removal of finished
  sequences so freed slots can be refilled ("Why Static Batching Wastes an RX
  9070 XT Agent Swarm", section "Continuous batching refills the slot instead
  of freezing it").

Readings where the pages are silent:

* Layer: pre-norm decoder layer, RMSNorm (eps 1e-6) with learned gains, no
  biases, rotate-half RoPE (theta 1e6) on q and k at absolute position, GQA
  with n_q / n_kv query heads per KV head, SwiGLU FFN, final RMSNorm, untied
  LM head, temperature 1.
* Storage points: weights, embeddings and the KV cache are bf16, so K and V
  of every verified row are rounded to bf16 (round to nearest even) when they
  enter the cache, and the final normed row is rounded to bf16 as the LM
  head's input.  Every other intermediate (q, the attention output, the
  residual stream, the norms, the SwiGLU product) is carried unrounded.
  Logits and probabilities are produced in float64 and returned as float32.
* Rows: row 0 of sequence b carries the last committed token at position L_b
  (not yet in the cache), row i the draft token i at position L_b + i; all
  gamma_b + 1 rows write K/V at their positions; row i attends to positions
  0 .. L_b + i.  p at row i judges draft token i+1; row gamma_b gives the
  bonus distribution.
* Acceptance of draft token x at row i: accept iff (p >= q and p > 0) or
  u*q < p, all in float32 (u < min(1, p/q) without a division; a token the
  target gives probability zero is never accepted).  u of row i (i < gamma_b)
  is the acceptance draw of draft i+1; u of row gamma_b is the draw of the
  final token (residual resample or bonus).
* Final-token sampling by inverse CDF on integer weights
  W_j = floor(w_j * 2^32) (w in float32), S = sum W, U = floor(u * 2^24),
  T = floor(S * U / 2^24), token = smallest j with W_0 + ... + W_j > T.
  w = max(0, p - q) after a rejection (falls back to p when that sums to
  zero), w = p for the bonus.
* Realignment: new_len = L + a + 1; each live sequence then holds exactly
  ceil((new_len + gamma_max + 1) / page) pages; surplus tail pages are pushed
  on the free stack in slot order, missing pages are popped from its top in
  slot order; a finished sequence (generated count reaching its limit)
  releases all its pages and its slot; survivors keep their relative order.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), as float64.

    bf16 keeps the float32 exponent and 7 fraction bits; from float64 (52
    fraction bits) that means rounding away the low 45 fraction bits.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64)
    low = np.uint64(45)
    lsb = (b >> low) & np.uint64(1)
    b = (b + (np.uint64((1 << 44) - 1) + lsb)) & ~np.uint64((1 << 45) - 1)
    return b.view(np.float64)


def round_bf16_other(x: np.ndarray, nearest: np.ndarray) -> np.ndarray:
    """The bf16 neighbour of x on the far side from its nearest bf16 value.

    bf16 is sign-magnitude, so the adjacent value away from zero has magnitude
    bits one higher and the one towards zero one lower; from zero the step
    goes to the smallest subnormal of x's sign.  A value that is itself bf16
    has no other neighbour and is returned unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    nearest = np.asarray(nearest, dtype=np.float64)
    bits = f64_to_bf16_bits(nearest).astype(np.int32)
    sign = bits & 0x8000
    mag = bits & 0x7FFF
    away = np.abs(x) > np.abs(nearest)
    step = np.where(away, mag + 1, mag - 1)
    out = np.where(nearest == 0, np.where(x < 0, 0x8001, 0x0001), sign | step)
    return np.where(x == nearest, nearest, bf16_to_f64(out.astype(np.uint16)))


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 values that are already bf16-representable -> uint16 bits."""
    return (np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def fp16_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dequant_int4_g32(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """int4 group-32 weights -> float64 [N, K]: w = scale * code.

    packed uint8 [N, K/2]: low nibble holds the even k, high nibble the odd
    k, each a two's complement code in [-8, 7]; scales fp16 [N, K/32], one
    per 32 consecutive k.
    """
    lo = (packed & 0x0F).astype(np.int64)
    hi = (packed >> 4).astype(np.int64)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    n, half = packed.shape
    codes = np.empty((n, 2 * half), dtype=np.float64)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    s = np.repeat(fp16_to_f64(scales), 32, axis=1)
    return codes * s


# ---------------------------------------------------------------------------
# layer pieces (float64)
# ---------------------------------------------------------------------------


def weight_rows(w, r0: int, r1: int) -> np.ndarray:
    """Rows r0..r1-1 of a projection (bf16 bits or (packed, scales)) as float64."""
    if isinstance(w, tuple):
        return dequant_int4_g32(w[0][r0:r1], w[1][r0:r1])
    return bf16_to_f64(w[r0:r1])


def linear(x: np.ndarray, w, chunk: int = 8192) -> np.ndarray:
    """y = x W^T.  x float64 [R, K]; W has one output feature per row."""
    n = w[0].shape[0] if isinstance(w, tuple) else w.shape[0]
    y = np.empty((x.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, chunk):
        r1 = min(n, r0 + chunk)
        y[:, r0:r1] = x @ weight_rows(w, r0, r1).T
    return y


def rmsnorm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain, per row."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gain


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of x [R, heads, d] at absolute positions pos [R].

    Pair (j, j + d/2) is rotated by angle pos * theta^(-2j/d).
    """
    d = x.shape[-1]
    half = d // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / d)
    ang = pos.astype(np.float64)[:, None] * inv_freq[None, :]       # [R, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a = x[..., :half]
    b = x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softmax(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def attention_one(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V for one query vector q [d] over keys K, V [n, d]."""
    d = q.shape[0]
    s = (K @ q) / math.sqrt(d)
    p = softmax(s)
    return p @ V


# ---------------------------------------------------------------------------
# paged KV cache access
# ---------------------------------------------------------------------------


def kv_slot(page_table_row: np.ndarray, pos: int, page: int):
    return int(page_table_row[pos // page]), pos % page


def gather_kv(kv_pool_f64: np.ndarray, page_table_row: np.ndarray, n: int, page: int):
    """K, V of positions 0..n-1 of one sequence: float64 [n_kv, n, d] each."""
    pos = np.arange(n)
    pages = page_table_row[pos // page]
    slots = pos % page
    kv = kv_pool_f64[pages, :, :, slots, :]          # [n, n_kv, 2, d]
    return kv[:, :, 0, :].transpose(1, 0, 2), kv[:, :, 1, :].transpose(1, 0, 2)


# ---------------------------------------------------------------------------
# the forward pass over all verify rows
# ---------------------------------------------------------------------------


def tree_depths(parents) -> list:
    """Depth of every node of a tree given each node's parent (node 0 the root,
    parent[0] = -1, parent[i] < i)."""
    depth = []
    for i, par in enumerate(parents):
        depth.append(0 if i == 0 else depth[int(par)] + 1)
    return depth


def tree_ancestors(parents, i: int) -> list:
    """Node i and its ancestors up to the root, in increasing index order."""
    out = [i]
    while i > 0:
        i = int(parents[i])
        out.append(i)
    return sorted(out)


def forward(dims: dict, weights, kv_pool_bits: np.ndarray, page_table: np.ndarray,
            seq_lens, draft_lens, tokens, eps: float = 1e-6, theta: float = 1e6,
            slots=None, flips=None, parents=None):
    """Target-model forward over every verify row of the selected slots.

    Returns a dict with logits and probs (float64 [rows, V]), kv_rows where
    kv_rows[(b, pos)] = (k bf16 values [n_kv, d], v [n_kv, d]) for every row
    written this step, the intermediates, and the three rounded quantities
    before rounding (k_pre, v_pre [rows, n_kv, d]; h3_pre [rows, H]).
    ``slots`` restricts the pass to some sequences (each sequence's rows
    depend only on its own cache, so a subset is exact).

    ``flips``: keys ("k" | "v", row, kv_head, j) or ("h3", row, j), row being
    the global row index; those bf16 roundings take the other neighbour of the
    exact value instead of the nearest one.  A value within the arithmetic
    error of a rounding tie may round either way in a finite-precision
    evaluation; this lets a caller reproduce such a choice.

    ``parents`` (token trees): [R] parent of every row within its sequence
    (-1 for row 0, the root; parent < own index).  Row i then sits at position
    L + depth(i) (its rotary angle) while its K/V goes to cache slot L + i, and
    it attends to the cached context and to its own ancestors and itself only.
    None: every sequence is a chain (row i's parent is row i - 1).
    """
    H, nq, nkv, d, P = dims["hidden"], dims["n_q"], dims["n_kv"], dims["head_dim"], dims["page"]
    seq_lens = np.asarray(seq_lens)
    draft_lens = np.asarray(draft_lens)
    B = len(seq_lens)
    offs = np.concatenate([[0], np.cumsum(draft_lens + 1)])
    if slots is None:
        slots = list(range(B))
    rows, row_seq, row_pos, row_slot, row_keys = [], [], [], [], []
    for b in slots:
        n_b = int(draft_lens[b]) + 1
        par = list(range(-1, n_b - 1)) if parents is None else \
            [int(x) for x in np.asarray(parents)[int(offs[b]): int(offs[b]) + n_b]]
        depth = tree_depths(par)
        L = int(seq_lens[b])
        for i in range(n_b):
            rows.append(int(offs[b]) + i)
            row_seq.append(b)
            row_pos.append(L + depth[i])
            row_slot.append(L + i)
            row_keys.append(list(range(L)) + [L + j for j in tree_ancestors(par, i)])
    rows = np.array(rows, dtype=np.int64)
    row_pos = np.array(row_pos, dtype=np.int64)
    tok = np.asarray(tokens)[rows]

    # embedding + attention pre-norm
    x0 = bf16_to_f64(weights.emb[tok])
    h1 = rmsnorm(x0, bf16_to_f64(weights.g_attn), eps)

    # fused QKV projection, RoPE on q and k; K and V enter the bf16 cache
    qkv = linear(h1, weights.proj["qkv"])
    q = qkv[:, : nq * d].reshape(-1, nq, d)
    k = qkv[:, nq * d: (nq + nkv) * d].reshape(-1, nkv, d)
    v = qkv[:, (nq + nkv) * d:].reshape(-1, nkv, d)
    q = rope(q, row_pos, theta)
    k_pre = rope(k, row_pos, theta)
    v_pre = v
    k = round_bf16(k_pre)
    v = round_bf16(v_pre)
    local = {int(r): n for n, r in enumerate(rows)}
    for key in (flips or ()):
        if key[0] in ("k", "v") and int(key[1]) in local:
            n, hk, j = local[int(key[1])], int(key[2]), int(key[3])
            tgt, pre = (k, k_pre) if key[0] == "k" else (v, v_pre)
            tgt[n, hk, j] = round_bf16_other(pre[n, hk, j], tgt[n, hk, j])

    # every row's K/V goes into its sequence's pages at its position
    kv_rows = {}
    kv_seq = {}
    for n, b in enumerate(row_seq):
        kv_rows[(b, int(row_slot[n]))] = (k[n], v[n])
    for b in slots:
        L = int(seq_lens[b])
        n_total = L + int(draft_lens[b]) + 1
        pool_rows = page_table[b]
        Kc = np.zeros((nkv, n_total, d))
        Vc = np.zeros((nkv, n_total, d))
        # cached positions 0..L-1 come from the pool
        if L > 0:
            pos = np.arange(L)
            pg = pool_rows[pos // P]
            sl = pos % P
            sub = kv_pool_bits[pg, :, :, sl, :]                  # [L, n_kv, 2, d]
            Kc[:, :L] = bf16_to_f64(sub[:, :, 0, :]).transpose(1, 0, 2)
            Vc[:, :L] = bf16_to_f64(sub[:, :, 1, :]).transpose(1, 0, 2)
        for i in range(int(draft_lens[b]) + 1):
            kk, vv = kv_rows[(b, L + i)]
            Kc[:, L + i] = kk
            Vc[:, L + i] = vv
        kv_seq[b] = (Kc, Vc)

    # block-causal GQA attention: a row sees the cached context and the rows of
    # its own draft block on its path from the root (for a chain: positions 0..t)
    group = nq // nkv
    o = np.zeros((len(rows), nq, d))
    for n, b in enumerate(row_seq):
        Kc, Vc = kv_seq[b]
        keys = np.array(row_keys[n], dtype=np.int64)
        for h in range(nq):
            g = h // group
            o[n, h] = attention_one(q[n, h], Kc[g][keys], Vc[g][keys])
    o = o.reshape(len(rows), nq * d)

    # output projection + residual
    x1 = x0 + linear(o, weights.proj["o"])
    # FFN pre-norm, SwiGLU, down projection + residual
    h2 = rmsnorm(x1, bf16_to_f64(weights.g_ffn), eps)
    gate = linear(h2, weights.proj["gate"])
    up = linear(h2, weights.proj["up"])
    act = silu(gate) * up
    x2 = x1 + linear(act, weights.proj["down"])
    # final norm (bf16 LM-head input) + LM head + softmax
    h3_pre = rmsnorm(x2, bf16_to_f64(weights.g_final), eps)
    h3 = round_bf16(h3_pre)
    for key in (flips or ()):
        if key[0] == "h3" and int(key[1]) in local:
            n, j = local[int(key[1])], int(key[2])
            h3[n, j] = round_bf16_other(h3_pre[n, j], h3[n, j])
    logits = linear(h3, weights.w_lm)
    probs = softmax(logits)
    return dict(rows=rows, logits=logits, probs=probs, kv_rows=kv_rows,
                h1=h1, q=q, o=o, x1=x1, act=act, x2=x2, h3=h3,
                k_pre=k_pre, v_pre=v_pre, h3_pre=h3_pre)


# ---------------------------------------------------------------------------
# acceptance and final-token sampling (float32 decisions, integer sampling)
# ---------------------------------------------------------------------------


def accepts(p: np.float32, q: np.float32, u: np.float32) -> bool:
    """Leviathan acceptance u < min(1, p/q), evaluated without a division."""
    p = np.float32(p)
    q = np.float32(q)
    u = np.float32(u)
    return bool((p >= q and p > np.float32(0)) or (np.float32(u * q) < p))


def inverse_cdf_int(w: np.ndarray, u: np.float32) -> int:
    """Index drawn from weights w (float32 [V]) with one uniform u, on integers.

    W_j = floor(w_j * 2^32); S = sum W; T = floor(S * floor(u * 2^24) / 2^24);
    returns the smallest j with W_0 + ... + W_j > T (or -1 when S == 0).
    """
    w = np.asarray(w, dtype=np.float32)
    W = np.floor(w.astype(np.float64) * 4294967296.0).astype(np.uint64)
    cum = np.cumsum(W, dtype=np.uint64)
    S = int(cum[-1])
    if S == 0:
        return -1
    U = int(math.floor(float(np.float32(u)) * 16777216.0))
    T = (S * U) >> 24
    return int(np.searchsorted(cum, np.uint64(T), side="right"))


def accept_and_sample(p_rows: np.ndarray, q_rows: np.ndarray, drafts, u: np.ndarray):
    """One sequence: (accepted count a, final token t).

    p_rows float32 [gamma+1, V] (target distribution at each verify row),
    q_rows float32 [gamma, V] (draft distribution each draft was proposed
    from), drafts [gamma] (draft tokens 1..gamma), u float32 [gamma+1].
    """
    gamma = len(drafts)
    p_rows = np.asarray(p_rows, dtype=np.float32)
    q_rows = np.asarray(q_rows, dtype=np.float32)
    a = gamma
    for i in range(gamma):
        x = int(drafts[i])
        if not accepts(p_rows[i, x], q_rows[i, x], u[i]):
            a = i
            break
    if a < gamma:
        w = np.maximum(np.float32(0), p_rows[a] - q_rows[a])
        if not np.any(np.floor(w.astype(np.float64) * 4294967296.0) > 0):
            w = p_rows[a]
    else:
        w = p_rows[gamma]
    t = inverse_cdf_int(w, u[gamma])
    return a, t


def greedy_accept(rows: np.ndarray, drafts):
    """Greedy verification of one sequence (temperature -> 0): draft i + 1 is kept
    iff it is the argmax of row i, the first draft that is not ends the prefix,
    and the final token is the argmax of the row after the kept prefix (the
    target's own next token).  Argmax = the smallest index among equal maxima.
    rows: [gamma + 1, V] (probabilities or logits: the same argmax).
    """
    gamma = len(drafts)
    a = gamma
    for i in range(gamma):
        if int(drafts[i]) != int(np.argmax(rows[i])):
            a = i
            break
    return a, int(np.argmax(rows[a]))


def greedy_tree_accept(rows: np.ndarray, node_tokens, parents):
    """Greedy verification of one sequence's token tree: from the root, descend
    into the child whose token is the argmax of the current node's row (the
    smallest such child index if several), as long as there is one; the final
    token is the argmax at the node reached.  rows [T, V] (logits or
    probabilities), node_tokens [T] (node 0 the root), parents [T].
    Returns (accepted count = depth reached, final token, path of node indices
    at depths 1..a)."""
    T = len(parents)
    v, path = 0, []
    while True:
        want = int(np.argmax(rows[v]))
        kids = [c for c in range(1, T) if int(parents[c]) == v and int(node_tokens[c]) == want]
        if not kids:
            break
        v = kids[0]
        path.append(v)
    return len(path), int(np.argmax(rows[v])), path


def accept_batch(p: np.ndarray, q: np.ndarray, tokens, uniforms, draft_lens, greedy: bool = False,
                 parents=None):
    """Every sequence of a batch: accepted counts, emitted tokens, emitted offsets.

    p float32 [R, V], q float32 [G, V]; emitted tokens of sequence b are its
    accepted drafts followed by its final token, packed at
    offset sum_{j<b}(a_j + 1).  greedy: the argmax rule of greedy_accept
    (q and uniforms are not read).
    """
    draft_lens = np.asarray(draft_lens)
    B = len(draft_lens)
    roff = np.concatenate([[0], np.cumsum(draft_lens + 1)])
    goff = np.concatenate([[0], np.cumsum(draft_lens)])
    acc = np.zeros(B, dtype=np.int32)
    fin = np.zeros(B, dtype=np.int32)
    paths = []
    for b in range(B):
        g = int(draft_lens[b])
        r0 = int(roff[b])
        drafts = np.asarray(tokens)[r0 + 1: r0 + 1 + g]
        if parents is not None:
            if not greedy:
                raise ValueError("token trees are verified greedily")
            a, t, path = greedy_tree_accept(p[r0: r0 + g + 1], np.asarray(tokens)[r0: r0 + g + 1],
                                            np.asarray(parents)[r0: r0 + g + 1])
            paths.append(path)
        elif greedy:
            a, t = greedy_accept(p[r0: r0 + g + 1], drafts)
        else:
            a, t = accept_and_sample(p[r0: r0 + g + 1], q[int(goff[b]): int(goff[b]) + g],
                                     drafts, np.asarray(uniforms, dtype=np.float32)[r0: r0 + g + 1])
        acc[b] = a
        fin[b] = t
    eoff = np.concatenate([[0], np.cumsum(acc.astype(np.int64) + 1)]).astype(np.int32)
    emitted = np.zeros(int(eoff[-1]), dtype=np.int32)
    for b in range(B):
        r0 = int(roff[b])
        a = int(acc[b])
        nodes = [r0 + c for c in paths[b]] if parents is not None else list(range(r0 + 1, r0 + 1 + a))
        emitted[eoff[b]: eoff[b] + a] = np.asarray(tokens)[nodes]
        emitted[eoff[b] + a] = fin[b]
    if parents is not None:
        return acc, emitted, eoff, fin, paths
    return acc, emitted, eoff, fin


def accept_histogram(acc, draft_lens, gamma_max: int):
    """Per draft position k: how many sequences tested it, how many accepted it.

    Position k (0-based) is tested when gamma_b > k and the k earlier drafts
    were accepted; the conditional acceptance at k is accepted/tested
    ("High Batch Size" post, section "How do you measure this on your own
    server?").
    """
    tested = np.zeros(gamma_max, dtype=np.int64)
    accepted = np.zeros(gamma_max, dtype=np.int64)
    for a, g in zip(acc, draft_lens):
        for k in range(int(g)):
            if a >= k:
                tested[k] += 1
            if a > k:
                accepted[k] += 1
    return tested, accepted


# ---------------------------------------------------------------------------
# realignment: lengths, pages, free stack, slots
# ---------------------------------------------------------------------------

OK = 0
ERR_CAPACITY = 2


def realign(seq_lens, accepted, page_table, num_pages, free_pages, num_free: int,
            page: int, gamma_max: int, gen_counts=None, gen_limits=None):
    """Realign every slot from its own accepted count.

    Returns a dict with new_seq_lens, finished, new_gen_counts, page_table,
    num_pages, free_pages, num_free (after the page moves) and the compacted
    next-slot view (src slot per new slot, and the per-slot arrays gathered
    through it), plus a status code.  On a capacity error nothing moves.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    accepted = np.asarray(accepted, dtype=np.int64)
    B = len(seq_lens)
    pt = np.array(page_table, dtype=np.int32, copy=True)
    npg = np.array(num_pages, dtype=np.int32, copy=True)
    fp = np.array(free_pages, dtype=np.int32, copy=True)
    max_pages = pt.shape[1]

    new_len = seq_lens + accepted + 1
    if gen_counts is not None and gen_limits is not None:
        new_gen = np.asarray(gen_counts, dtype=np.int64) + accepted + 1
        finished = new_gen >= np.asarray(gen_limits, dtype=np.int64)
    else:
        new_gen = None if gen_counts is None else np.asarray(gen_counts, dtype=np.int64) + accepted + 1
        finished = np.zeros(B, dtype=bool)

    need = np.where(finished, 0, (new_len + gamma_max + 1 + page - 1) // page)
    status = OK
    if np.any(need > max_pages):
        status = ERR_CAPACITY
    surplus = np.maximum(0, npg - need)
    deficit = np.maximum(0, need - npg)
    top_after_push = num_free + int(surplus.sum())
    if int(deficit.sum()) > top_after_push:
        status = ERR_CAPACITY

    out = dict(status=status, new_seq_lens=new_len.astype(np.int32),
               finished=finished.astype(np.int32),
               new_gen_counts=None if new_gen is None else new_gen.astype(np.int32))
    if status != OK:
        out.update(page_table=np.array(page_table, dtype=np.int32, copy=True),
                   num_pages=np.array(num_pages, dtype=np.int32, copy=True),
                   free_pages=np.array(free_pages, dtype=np.int32, copy=True),
                   num_free=num_free)
        return out

    # push every slot's surplus tail pages, slot by slot, low logical page first
    stack = list(fp[:num_free])
    for b in range(B):
        for j in range(int(need[b]), int(npg[b])):
            stack.append(int(pt[b, j]))
            pt[b, j] = -1
    # pop the missing pages from the top, slot by slot
    for b in range(B):
        for j in range(int(npg[b]), int(need[b])):
            pt[b, j] = stack.pop()
    npg = need.astype(np.int32)
    new_fp = np.array(fp, copy=True)
    new_fp[: len(stack)] = np.array(stack, dtype=np.int32)

    # stable compaction of the surviving slots
    src = np.array([b for b in range(B) if not finished[b]], dtype=np.int32)
    out.update(page_table=pt, num_pages=npg, free_pages=new_fp, num_free=len(stack),
               next_src=src, num_live=len(src),
               next_seq_lens=new_len[src].astype(np.int32),
               next_num_pages=npg[src].astype(np.int32),
               next_page_table=pt[src],
               next_gen_counts=None if new_gen is None else new_gen[src].astype(np.int32))
    return out


# ---------------------------------------------------------------------------
# admission: the refill half of continuous batching
# ---------------------------------------------------------------------------
# "Why Static Batching Wastes an RX 9070 XT Agent Swarm and Continuous
# Batching Wins It Back", section "Continuous batching refills the slot
# instead of freezing it": a slot freed by a finished sequence takes a waiting
# one on the very next step, so the batch stays full while work is queued.
# The pages say nothing about memory; the reading here: a newcomer arrives
# with its context already cached (prefill is charged outside the step) and
# must get the pages of its context plus one step of drafts; it is admitted,
# in arrival order, while a slot is free and the free pages cover it plus one
# step of growth for every sequence live after it, so the next realignment
# can never run out of pages.

ERR_BAD_INPUT = 6


def pages_for(length: int, gamma_max: int, page: int) -> int:
    """Pages a sequence of `length` cached positions holds: room for one more
    verify block of gamma_max + 1 rows."""
    return -(-(int(length) + gamma_max + 1) // page)


def admission_count(queue_ctx, live: int, free_pages: int, slots: int, gamma_max: int, page: int) -> int:
    """How many queued sequences (contexts in arrival order) enter this step.

    Newcomer n (0-based) is admitted when live + n < slots and
    pages_for(L_n) + (live + n + 1) * ceil((gamma_max + 1) / page) does not
    exceed the free pages left after newcomers 0 .. n-1; the first one that
    fails stops the admission, so arrival order is never overtaken."""
    growth = -(-(gamma_max + 1) // page)
    free = int(free_pages)
    n = 0
    for L in queue_ctx:
        if live + n >= slots:
            break
        need = pages_for(L, gamma_max, page)
        if need + (live + n + 1) * growth > free:
            break
        free -= need
        n += 1
    return n


def admit(table: dict, live: int, ctx_lens, out_lens, free_pages, num_free: int, gamma_max: int, page: int,
          num_live=None, next_src=None, gen_limits_prev=None):
    """Append admitted sequences to a slot table (the device half of admission).

    ``table``: seq_lens, num_pages, gen_counts, gen_limits [slots] and
    page_table [slots, max_pages], with the survivors of the last
    realignment at slots 0 .. live-1.  When ``next_src`` and
    ``gen_limits_prev`` are given, the survivors' output lengths are first
    gathered from the table before the compaction.  Newcomer j goes to slot
    live + j with length ctx_lens[j], generated count 0, output length
    out_lens[j] and pages_for(ctx_lens[j]) pages popped from the top of the
    free stack (``free_pages[:num_free]``, top last) in admission order:
    newcomer j's k-th page is the (sum of earlier newcomers' pages + k)-th
    page popped; the rest of its row is -1.

    Returns (status, new table, new num_free).  Errors (nothing changes):
    num_live given and != live, or a negative context (ERR_BAD_INPUT); a row
    wider than max_pages, or more pages than the stack holds (ERR_CAPACITY).
    """
    t = {k: np.array(v, copy=True) for k, v in table.items()}
    max_pages = t["page_table"].shape[1]
    ctx_lens = [int(x) for x in ctx_lens]
    need = [pages_for(L, gamma_max, page) for L in ctx_lens]
    if num_live is not None and int(num_live) != live:
        return ERR_BAD_INPUT, t, num_free
    if any(L < 0 for L in ctx_lens):
        return ERR_BAD_INPUT, t, num_free
    if any(n > max_pages for n in need) or sum(need) > num_free:
        return ERR_CAPACITY, t, num_free
    if next_src is not None and gen_limits_prev is not None:
        for j in range(live):
            t["gen_limits"][j] = gen_limits_prev[int(next_src[j])]
    top = int(num_free)
    for j, (L, out) in enumerate(zip(ctx_lens, out_lens)):
        s = live + j
        t["seq_lens"][s] = L
        t["num_pages"][s] = need[j]
        t["gen_counts"][s] = 0
        t["gen_limits"][s] = int(out)
        t["page_table"][s, :] = -1
        for k in range(need[j]):
            top -= 1
            t["page_table"][s, k] = free_pages[top]
    return OK, t, top


# ---------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------


def compact_kv(pool_bits: np.ndarray, page_table, seq_lens, paths, page: int) -> np.ndarray:
    """After a token tree's verification: the K/V of the node at depth k of
    sequence b's accepted path moves from cache slot L_b + node to slot L_b + k,
    so the accepted tokens sit at consecutive positions (a chain's path is
    already in place).  Returns the moved pool (bf16 bits)."""
    out = np.array(pool_bits, copy=True)
    for b, path in enumerate(paths):
        L = int(seq_lens[b])
        for k, node in enumerate(path, start=1):
            src, dst = L + int(node), L + k
            if src == dst:
                continue
            ps, pd = page_table[b][src // page], page_table[b][dst // page]
            out[pd, :, :, dst % page, :] = pool_bits[ps, :, :, src % page, :]
    return out


def verify_step(batch, weights, eps: float = 1e-6, theta: float = 1e6, slots=None, greedy: bool = False,
                parents=None):
    """Forward, acceptance, sampling and realignment of one batch.

    ``batch`` and ``weights`` are the seeded inputs (workloads.Batch /
    workloads.Weights).  With ``slots`` the forward, acceptance and sampling
    run for those sequences only (realignment is skipped).  ``greedy``:
    greedy verification on the float64 logits (greedy_accept).
    """
    dims = batch.dims
    fw = forward(dims, weights, batch.kv_pool, batch.page_table, batch.seq_lens,
                 batch.draft_lens, batch.tokens, eps=eps, theta=theta, slots=slots, parents=parents)
    p32 = fw["probs"].astype(np.float32)
    out = dict(forward=fw, logits=fw["logits"], probs=fw["probs"], rows=fw["rows"])
    if slots is not None:
        # per-sequence acceptance for the chosen slots
        roff = np.concatenate([[0], np.cumsum(batch.draft_lens + 1)])
        goff = np.concatenate([[0], np.cumsum(batch.draft_lens)])
        res = {}
        n = 0
        for b in slots:
            g = int(batch.draft_lens[b])
            r0 = int(roff[b])
            a, t = accept_and_sample(p32[n: n + g + 1],
                                     batch.draft_probs[int(goff[b]): int(goff[b]) + g],
                                     batch.tokens[r0 + 1: r0 + 1 + g],
                                     batch.uniforms[r0: r0 + g + 1])
            res[b] = (a, t)
            n += g + 1
        out["per_slot"] = res
        return out
    if parents is not None:
        acc, emitted, eoff, fin, paths = accept_batch(fw["logits"], None, batch.tokens, None, batch.draft_lens,
                                                      greedy=True, parents=parents)
        out["paths"] = paths
    else:
        acc, emitted, eoff, fin = accept_batch(fw["logits"] if greedy else p32, batch.draft_probs, batch.tokens,
                                               batch.uniforms, batch.draft_lens, greedy=greedy)
    ra = realign(batch.seq_lens, acc, batch.page_table, batch.num_pages, batch.free_pages,
                 batch.num_free, dims["page"], batch.gamma_max,
                 gen_counts=batch.gen_counts, gen_limits=batch.gen_limits)
    out.update(accepted=acc, emitted_tokens=emitted, emitted_offsets=eoff, final_tokens=fin,
               realign=ra)
    return out
