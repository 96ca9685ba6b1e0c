"""Seeded synthetic inputs for the ragged batched speculative-verify step.

This module is shared by the CPU oracle, the GPU parity tests and the bench.
It only draws random numbers and encodes them into the storage formats the
step consumes (bf16 bits, fp16 bits, packed int4); it contains none of the
verify step's arithmetic.

Random numbers come from numpy's Philox4x32-10 bit generator (Salmon et al.,
"Parallel random numbers: as easy as 1, 2, 3", SC'11), keyed by
``(0x5D5EED00 + workload index) << 8 | stream`` so that every workload and
every kind of input (weights, KV, tokens, q, u, per-sequence draws) has a
stream of its own.

Workload shapes follow the pages' setting: a single decoder layer of a 9B
class model (hidden 4096, 32 query / 8 KV heads of 128, SwiGLU FFN 12288,
vocab 151936) verified against ragged draft blocks, with the draft lengths,
context lengths and acceptance mixes the pages discuss ("Speculative Decoding
and Batching Compete for the Same Compute Slack on RDNA4", section "The budget
is fixed, and the batch is inside it"; "Speculative Decoding at High Batch
Size", section "What does one speculative iteration actually cost?"; the
splicedso primer, section "When it works").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# ---------------------------------------------------------------------------
# model dimensions
# ---------------------------------------------------------------------------

TINY = dict(hidden=256, n_q=4, n_kv=2, head_dim=64, ffn=768, vocab=1024, page=16)
NINE_B = dict(hidden=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288, vocab=151936, page=16)

RMS_EPS = 1e-6
ROPE_THETA = 1.0e6

# stream ids inside one workload key
S_WEIGHTS, S_KV, S_TOKENS, S_Q, S_U, S_SEQ = range(6)


def rng(workload: int, stream: int, sub: int = 0) -> np.random.Generator:
    """Philox generator for (workload, stream, sub-stream)."""
    return np.random.Generator(np.random.Philox(key=_key(workload, stream, sub)))


# ---------------------------------------------------------------------------
# storage encodings (inputs only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Encode float32 values as bf16 bit patterns (round to nearest, ties to even)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (b >> np.uint32(16)).astype(np.uint16)


def _key(workload: int, stream: int, sub: int = 0) -> int:
    return (((0x5D5EED00 + workload) << 8) | stream) << 32 | (sub & 0xFFFFFFFF)


def normal_bf16(key: int, shape, std: float, mean: float = 0.0, chunk: int = 1 << 22) -> np.ndarray:
    """bf16 bits of N(mean, std^2) draws.

    The array is cut into chunks of ``chunk`` elements; chunk i is drawn from
    Philox(key) jumped i + 1 times (independent streams), so the values do not
    depend on how many threads fill the chunks.
    """
    from concurrent.futures import ThreadPoolExecutor
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    base = np.random.Philox(key=key)

    def fill(i):
        c0, c1 = i * chunk, min(n, (i + 1) * chunk)
        g = np.random.Generator(base.jumped(i + 1))
        x = g.standard_normal(size=c1 - c0, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if mean != 0.0:
            x += np.float32(mean)
        b = x.view(np.uint32)
        t = b >> np.uint32(16)
        np.bitwise_and(t, np.uint32(1), out=t)
        np.add(t, np.uint32(0x7FFF), out=t)
        np.add(b, t, out=b)
        np.right_shift(b, np.uint32(16), out=b)
        out[c0:c1] = b

    nchunks = (n + chunk - 1) // chunk
    if nchunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(max_workers=min(16, nchunks)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def uniform24(g: np.random.Generator, n: int) -> np.ndarray:
    """fp32 uniforms on the 24-bit grid k / 2^24, k uniform in [0, 2^24)."""
    k = g.integers(0, 1 << 24, size=n, dtype=np.int64)
    return (k.astype(np.float64) / float(1 << 24)).astype(np.float32)


def softmax_f32(logits: np.ndarray) -> np.ndarray:
    """Input recipe for draft distributions: q = softmax(N(0, sigma) logits)."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


# ---------------------------------------------------------------------------
# weights
# ---------------------------------------------------------------------------

@dataclass
class Weights:
    """One decoder layer + embedding + LM head.

    bf16 tensors are uint16 bit arrays.  Layer projections are either bf16
    ``[N, K]`` (row n holds output feature n) or int4 group-32: ``packed``
    uint8 ``[N, K/2]`` (low nibble = even k, signed two's complement in
    [-8, 7]) and ``scales`` fp16 bits ``[N, K/32]`` (one per 32 consecutive k).
    Row order of the fused QKV projection: the n_q query heads, then the
    n_kv key heads, then the n_kv value heads, head_dim rows each.
    """
    dims: dict
    fmt: str                      # "bf16" or "int4"
    emb: np.ndarray               # bf16 [V, H]
    g_attn: np.ndarray            # bf16 [H]
    g_ffn: np.ndarray             # bf16 [H]
    g_final: np.ndarray           # bf16 [H]
    w_lm: np.ndarray              # bf16 [V, H]
    proj: dict = field(default_factory=dict)   # name -> bf16 [N,K] | (packed, scales)


PROJ_NAMES = ("qkv", "o", "gate", "up", "down")


def proj_shape(d: dict, name: str):
    H, F, hd = d["hidden"], d["ffn"], d["head_dim"]
    if name == "qkv":
        return ((d["n_q"] + 2 * d["n_kv"]) * hd, H)
    if name == "o":
        return (H, d["n_q"] * hd)
    if name in ("gate", "up"):
        return (F, H)
    if name == "down":
        return (H, F)
    raise KeyError(name)


def _int4_proj(g: np.random.Generator, n: int, k: int, std: float):
    """Random int4 codes uniform in [-8, 7] with fp16 scales giving ~std."""
    q = g.integers(-8, 8, size=(n, k), dtype=np.int8)
    # uniform on [-8,7] has std ~4.61; scale jitter keeps groups distinct
    s = (std / 4.61) * (0.75 + 0.5 * g.random(size=(n, k // 32), dtype=np.float32))
    scales = s.astype(np.float16).view(np.uint16)
    u = (q.astype(np.int16) & 0xF).astype(np.uint8)
    packed = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    return packed, scales


def make_weights(dims: dict, workload: int, fmt: str = "bf16", std: float = 0.02) -> Weights:
    H, V = dims["hidden"], dims["vocab"]
    sub = 0

    def nxt():
        nonlocal sub
        sub += 1
        return _key(workload, S_WEIGHTS, sub)

    emb = normal_bf16(nxt(), (V, H), std)
    # gains near one (not exactly one, so a dropped gain is visible)
    g_attn = normal_bf16(nxt(), (H,), 0.1, 1.0)
    g_ffn = normal_bf16(nxt(), (H,), 0.1, 1.0)
    g_final = normal_bf16(nxt(), (H,), 0.1, 1.0)
    w_lm = normal_bf16(nxt(), (V, H), std)
    proj = {}
    for name in PROJ_NAMES:
        n, k = proj_shape(dims, name)
        if fmt == "bf16":
            proj[name] = normal_bf16(nxt(), (n, k), std)
        elif fmt == "int4":
            proj[name] = _int4_proj(np.random.Generator(np.random.Philox(key=nxt())), n, k, std)
        else:
            raise ValueError(fmt)
    return Weights(dims=dims, fmt=fmt, emb=emb, g_attn=g_attn, g_ffn=g_ffn,
                   g_final=g_final, w_lm=w_lm, proj=proj)


# ---------------------------------------------------------------------------
# batch state: paged KV cache, page tables, draft blocks
# ---------------------------------------------------------------------------

@dataclass
class Batch:
    """Host copy of one verify step's inputs.

    KV pool layout: bf16 ``[num_pages, n_kv, 2 (K,V), page, head_dim]``.
    ``page_table[b, j]`` is the pool page holding positions
    ``j*page .. j*page+page-1`` of slot b's sequence; ``num_pages[b]`` entries
    are valid, the rest are -1.  ``free_pages[:num_free]`` is the free stack
    (top at the end).  Row layout: rows of slot b are contiguous starting at
    ``sum_{j<b}(gamma_j+1)``; row 0 carries the last committed token (not yet
    in the cache), rows 1..gamma_b the draft tokens.  ``draft_probs`` has one
    row per draft token: row ``sum_{j<b} gamma_j + i`` is the draft
    distribution q_i that draft token i+1 was proposed from.  ``uniforms`` has
    one value per verify row.
    """
    dims: dict
    gamma_max: int
    seq_lens: np.ndarray          # int32 [B]
    draft_lens: np.ndarray        # int32 [B]
    tokens: np.ndarray            # int32 [R]
    draft_probs: np.ndarray       # fp32 [G, V]
    uniforms: np.ndarray          # fp32 [R]
    kv_pool: np.ndarray           # bf16 bits [P, n_kv, 2, page, d]
    page_table: np.ndarray        # int32 [B, max_pages]
    num_pages: np.ndarray         # int32 [B]
    free_pages: np.ndarray        # int32 [P]
    num_free: int
    gen_counts: np.ndarray | None = None   # int32 [B]
    gen_limits: np.ndarray | None = None   # int32 [B]
    alphas: np.ndarray | None = None       # target acceptance per slot (recipe only)

    @property
    def B(self):
        return int(self.seq_lens.shape[0])

    @property
    def R(self):
        return int((self.draft_lens + 1).sum())

    @property
    def G(self):
        return int(self.draft_lens.sum())


def pages_needed(length: int, page: int) -> int:
    return (length + page - 1) // page


def make_batch(dims: dict, workload: int, seq_lens, draft_lens, gamma_max: int,
               extra_pages: int = 0, max_pages: int | None = None,
               q_sigma: float = 2.0, alphas=None, gen_limits=None,
               gen_counts=None, kv_fill: str = "normal") -> Batch:
    """Build a batch whose slots hold pages for L_b + gamma_max + 1 positions.

    Pages are taken from a shuffled pool so that page tables are not
    contiguous; ``extra_pages`` spare pages stay on the free stack.
    ``kv_fill="normal"`` fills every page with bf16 N(0,1); "lazy" leaves the
    pool zero (callers fill the used pages themselves).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    draft_lens = np.asarray(draft_lens, dtype=np.int32)
    B = seq_lens.shape[0]
    P, nkv, d, V = dims["page"], dims["n_kv"], dims["head_dim"], dims["vocab"]
    held = np.array([pages_needed(int(L) + gamma_max + 1, P) for L in seq_lens], dtype=np.int32)
    if max_pages is None:
        max_pages = int(held.max()) + 2
    total = int(held.sum()) + extra_pages
    g_seq = rng(workload, S_SEQ, 1)
    perm = g_seq.permutation(total).astype(np.int32)
    page_table = np.full((B, max_pages), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        page_table[b, :held[b]] = perm[o:o + held[b]]
        o += held[b]
    free = np.full(total, -1, dtype=np.int32)
    free[:extra_pages] = perm[o:]
    kv = np.zeros((total, nkv, 2, P, d), dtype=np.uint16)
    if kv_fill == "normal":
        fill_kv_normal(kv, workload)
    R = int((draft_lens + 1).sum())
    G = int(draft_lens.sum())
    tokens = rng(workload, S_TOKENS, 0).integers(0, V, size=R, dtype=np.int64).astype(np.int32)
    if G > 0:
        ql = rng(workload, S_Q, 0).standard_normal(size=(G, V), dtype=np.float32) * np.float32(q_sigma)
        draft_probs = softmax_f32(ql)
    else:
        draft_probs = np.zeros((0, V), dtype=np.float32)
    u = uniform24(rng(workload, S_U, 0), R)
    return Batch(dims=dims, gamma_max=gamma_max, seq_lens=seq_lens, draft_lens=draft_lens,
                 tokens=tokens, draft_probs=draft_probs, uniforms=u, kv_pool=kv,
                 page_table=page_table, num_pages=held, free_pages=free,
                 num_free=extra_pages,
                 gen_counts=None if gen_counts is None else np.asarray(gen_counts, np.int32),
                 gen_limits=None if gen_limits is None else np.asarray(gen_limits, np.int32),
                 alphas=None if alphas is None else np.asarray(alphas, np.float64))


def fill_kv_normal(kv: np.ndarray, workload: int, chunk: int = 512) -> None:
    """Fill a KV pool with bf16 N(0,1), one Philox sub-stream per chunk of pages."""
    for c0 in range(0, kv.shape[0], chunk):
        c1 = min(kv.shape[0], c0 + chunk)
        kv[c0:c1] = normal_bf16(_key(workload, S_KV, c0 // chunk), kv[c0:c1].shape, 1.0)


def row_offsets(draft_lens: np.ndarray) -> np.ndarray:
    """Exclusive prefix of (gamma_b + 1): first verify row of each slot (layout only)."""
    o = np.zeros(len(draft_lens) + 1, dtype=np.int64)
    o[1:] = np.cumsum(np.asarray(draft_lens, np.int64) + 1)
    return o


def retarget_draft_probs(batch: Batch, p_rows: np.ndarray, workload: int) -> None:
    """Input recipe: rebuild q so that draft token i+1 is accepted with prob alpha_b.

    Given the target distributions ``p_rows`` (fp32 [R, V], from a prepass of
    the forward), set q_i(x_{i+1}) = p_i(x_{i+1}) / alpha_b and rescale the
    other entries of q_i so the row sums to one.  Then min(1, p/q) = alpha_b
    exactly at every draft position (the pages' independent-acceptance model,
    "Speculative Decoding at High Batch Size", section "What does one
    speculative iteration actually cost?").
    """
    assert batch.alphas is not None
    offs = row_offsets(batch.draft_lens)
    q = batch.draft_probs.astype(np.float64)
    g_row = 0
    for b in range(batch.B):
        a = float(batch.alphas[b])
        for i in range(int(batch.draft_lens[b])):
            r = int(offs[b]) + i
            x = int(batch.tokens[r + 1])
            target = float(p_rows[r, x]) / a
            qi = q[g_row]
            rest = 1.0 - qi[x]
            qi *= (1.0 - target) / rest
            qi[x] = target
            g_row += 1
    batch.draft_probs = q.astype(np.float32)


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

WORKLOADS = {
    1: "tiny: B=2, gamma={3,1}, hidden 256, 4/2 heads of 64, FFN 768, vocab 1024, ctx 128",
    2: "batch-of-one: B=1, gamma=7, 9B-class layer bf16, vocab 151936, ctx 2048, alpha 0.8",
    3: "eight-agent ragged: B=8, gamma_b in {1,2,3} with sum<=16, ctx U{512..8192}, alpha in {0.97,0.8,0.14}",
    4: "crossover sweep: B in {1,4,16,32,64,128} x gamma in {0,1,2,3,4,7,8}, ctx 2048, alpha 0.8",
    5: "swarm: B=128 slots, int4 g32 layer, gamma_b=clamp((512-B)/B,0,3), ctx U{1024..16384}, outputs loguniform 40..900",
}

SWEEP_B = (1, 4, 16, 32, 64, 128)
SWEEP_GAMMA = (0, 1, 2, 3, 4, 7, 8)
ALPHA_MIX = (0.97, 0.8, 0.14)


def workload1(extra_pages: int = 8) -> Batch:
    return make_batch(TINY, 1, seq_lens=[128, 128], draft_lens=[3, 1], gamma_max=3,
                      extra_pages=extra_pages)


def workload2(**kw) -> Batch:
    return make_batch(NINE_B, 2, seq_lens=[2048], draft_lens=[7], gamma_max=7,
                      alphas=[0.8], **kw)


def workload3_shape(workload: int = 3):
    g = rng(workload, S_SEQ, 0)
    while True:
        gam = g.integers(1, 4, size=8)
        if gam.sum() <= 16:
            break
    lens = g.integers(512, 8193, size=8)
    alphas = np.array(ALPHA_MIX)[g.integers(0, 3, size=8)]
    return lens.astype(np.int32), gam.astype(np.int32), alphas


def workload3(**kw) -> Batch:
    lens, gam, alphas = workload3_shape()
    return make_batch(NINE_B, 3, seq_lens=lens, draft_lens=gam, gamma_max=3,
                      alphas=alphas, **kw)


def workload4(B: int, gamma: int, **kw) -> Batch:
    return make_batch(NINE_B, 4, seq_lens=[2048] * B, draft_lens=[gamma] * B,
                      gamma_max=max(gamma, 1), alphas=[0.8] * B, **kw)


def swarm_gamma(live: int, budget: int = 512, cap: int = 3) -> int:
    """Adaptive draft length: (budget - B) / B, clamped to [0, cap]."""
    if live <= 0:
        return 0
    return int(max(0, min(cap, (budget - live) // live)))


def loguniform_lengths(g: np.random.Generator, n: int, lo: int = 40, hi: int = 900) -> np.ndarray:
    return np.floor(np.exp(g.uniform(math.log(lo), math.log(hi), size=n))).astype(np.int32)


def workload5_shape(workload: int = 5, B: int = 128):
    g = rng(workload, S_SEQ, 0)
    lens = g.integers(1024, 16385, size=B).astype(np.int32)
    alphas = np.array(ALPHA_MIX)[g.integers(0, 3, size=B)]
    limits = loguniform_lengths(g, B)
    gam = np.full(B, swarm_gamma(B), dtype=np.int32)
    return lens, gam, alphas, limits


def swarm_requests(n: int, workload: int = 5, ctx=(1024, 16384), outs=(40, 900)):
    """The swarm's arrival queue: n sequences with context U{ctx}, output length
    log-uniform in outs, and a target acceptance from ALPHA_MIX (recipe only)."""
    g = rng(workload, S_SEQ, 7)
    lens = g.integers(ctx[0], ctx[1] + 1, size=n).astype(np.int32)
    limits = loguniform_lengths(g, n, *outs)
    alphas = np.array(ALPHA_MIX)[g.integers(0, 3, size=n)]
    return lens, limits, alphas
