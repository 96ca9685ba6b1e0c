"""Greedy verification on the GPU (sdv_set_sampling(GREEDY)) against the oracle,
through the C ABI: bit-exact on given probabilities (ties included), and whole
steps on the tiny and 9B-class models with drafts planted from the oracle's own
argmax chain, so that sequences accept none, some or all of their drafts."""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
GREEDY = 1


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available()
    return torch


def _given_probs_case(dims, B, gmax, seed):
    g = np.random.default_rng(seed)
    V = dims["vocab"]
    gam = g.integers(0, gmax + 1, size=B)
    lens = g.integers(0, 300, size=B)
    b = wl.make_batch(dims, 950 + seed, seq_lens=lens, draft_lens=gam, gamma_max=gmax, extra_pages=3 * B,
                      kv_fill="lazy")
    p = wl.softmax_f32(g.standard_normal((b.R, V)).astype(np.float32) * 2)
    roff = wl.row_offsets(b.draft_lens)
    for s in range(B):
        for i in range(int(gam[s])):
            r = int(roff[s]) + i
            kind = (s + i) % 4
            if kind in (0, 1):
                b.tokens[r + 1] = int(np.argmax(p[r]))          # the target's own token: kept
            if kind == 2:
                # the draft ties for the maximum: the smaller index is the argmax
                # (a draft above 0 loses to a smaller twin, a draft 0 wins against 1)
                x = int(b.tokens[r + 1])
                y = x // 2 if x > 0 else 1
                top = np.float32(p[r].max() * 1.5)
                p[r, x] = top
                p[r, y] = top
    return b, p


@pytest.mark.parametrize("dims,B,gmax,seed", [(wl.TINY, 9, 3, 0), (wl.TINY, 64, 7, 1), (wl.NINE_B, 5, 7, 2)])
def test_greedy_accept_bit_exact(torch_cuda, dims, B, gmax, seed):
    import torch
    from workloads import device as wd
    b, p = _given_probs_case(dims, B, gmax, seed)
    W = wl.make_weights(wl.TINY, 1)
    if dims is wl.NINE_B:
        from tests.test_gpu_parity import _attn_only_engine
        eng = _attn_only_engine(wd.config(dims, gmax), torch)
    else:
        eng = gh.engine_for(dims, gmax, wd.weights_to_device(W), max(b.R, 16), 128)
    eng.set_sampling(GREEDY)
    bd = wd.batch_to_device(b)
    bd["draft_probs"] = None   # greedy verification reads neither q nor u
    bd["uniforms"] = None
    res = wd.alloc_result(b.B, b.R, dims["vocab"], gmax, b.page_table.shape[1])
    eng.accept(torch.from_numpy(p).cuda(), bd, res)
    assert eng.read_status(res["status"]) == 0
    acc, emitted, eoff, fin = o.accept_batch(p, None, b.tokens, None, b.draft_lens, greedy=True)
    c = lambda k: res[k].cpu().numpy()  # noqa: E731
    assert np.array_equal(c("accepted"), acc)
    assert np.array_equal(c("final_tokens"), fin)
    assert np.array_equal(c("emitted_offsets"), eoff)
    assert np.array_equal(c("emitted_tokens")[:eoff[-1]], emitted)
    ra = o.realign(b.seq_lens, acc, b.page_table, b.num_pages, b.free_pages, b.num_free, dims["page"], gmax)
    assert np.array_equal(bd["page_table"].cpu().numpy(), ra["page_table"])
    assert acc.max() > 0 and (acc < b.draft_lens).any()


def _plant_argmax_drafts(batch, W, plan):
    """plan[b] = how many leading drafts of sequence b to set to the oracle's argmax
    (drafts after them stay random).  Each planted draft needs the forward of the
    drafts before it, so the oracle runs once per planted position."""
    roff = wl.row_offsets(batch.draft_lens)
    for depth in range(max(plan) if len(plan) else 0):
        fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens,
                       batch.tokens)
        for s, k in enumerate(plan):
            if depth < k:
                r = int(roff[s]) + depth
                batch.tokens[r + 1] = int(np.argmax(fw["logits"][r]))


def _check_greedy_step(eng, W, batch, name):
    status, res, dev = gh.run_step(eng, batch)
    assert status == 0, f"{name}: status {status}"
    ref = o.verify_step(batch, W, greedy=True)
    z = ref["logits"]
    tol = 1e-2 * np.sqrt(np.mean(z ** 2))
    assert np.abs(res["logits"] - z).max() <= tol, name
    top2 = np.sort(z, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 2 * tol     # the GPU's argmax must equal the oracle's here
    roff = wl.row_offsets(batch.draft_lens)
    judged = 0
    for s in range(batch.B):
        g, r0 = int(batch.draft_lens[s]), int(roff[s])
        a_ref = int(ref["accepted"][s])
        # every slot: each token the GPU kept or drew is within the logit tolerance
        # of the oracle's maximum at its row, and it stopped at a draft that
        # differs from the token it drew there
        a_g = int(res["accepted"][s])
        chosen = [int(x) for x in batch.tokens[r0 + 1: r0 + 1 + a_g]] + [int(res["final_tokens"][s])]
        for i, tok in enumerate(chosen):
            assert z[r0 + i, tok] >= z[r0 + i].max() - 2 * tol, (name, s, i, tok)
        if a_g < g:
            assert int(batch.tokens[r0 + 1 + a_g]) != chosen[-1], (name, s)
        # every decision row up to and including the final one must be clear
        if not clear[r0: r0 + min(a_ref, g) + 1].all():
            continue
        assert int(res["accepted"][s]) == a_ref, (name, s)
        assert int(res["final_tokens"][s]) == int(ref["final_tokens"][s]), (name, s)
        judged += 1
    assert judged >= batch.B // 2, (name, judged)
    # realignment from the GPU's own counts and tokens, bit-exact, always
    gh.check_realign(batch, res, dev)
    return ref


def test_greedy_step_tiny(torch_cuda):
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1)
    eng = gh.engine_for(wl.TINY, 4, wd.weights_to_device(W), 64, 16)
    eng.set_sampling(GREEDY)
    lens = [128, 7, 60, 200, 0, 33]
    gam = [4, 3, 4, 2, 1, 4]
    batch = wl.make_batch(wl.TINY, 61, seq_lens=lens, draft_lens=gam, gamma_max=4, extra_pages=8)
    plan = [4, 0, 2, 2, 1, 3]   # all kept (bonus), none, partial, all, all, partial
    _plant_argmax_drafts(batch, W, plan)
    ref = _check_greedy_step(eng, W, batch, "tiny-greedy")
    # the oracle keeps exactly the planted drafts (a random draft after them is rejected)
    assert ref["accepted"].tolist() == plan


def test_greedy_step_nine_b(torch_cuda, nine_b_weights):
    W, Wd = nine_b_weights
    eng = gh.engine_for(wl.NINE_B, 3, Wd, 32, 8)
    eng.set_sampling(GREEDY)
    batch = wl.make_batch(wl.NINE_B, 62, seq_lens=[2048, 513, 1000], draft_lens=[3, 2, 0], gamma_max=3,
                          extra_pages=8)
    _plant_argmax_drafts(batch, W, [2, 1, 0])
    ref = _check_greedy_step(eng, W, batch, "nine-b-greedy")
    assert int(ref["accepted"][0]) >= 2 and int(ref["accepted"][1]) >= 1
