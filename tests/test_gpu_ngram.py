"""n-gram drafts with greedy verification on the GPU (tiny model, through the C
ABI): speculating with drafts copied from each sequence's own history emits
exactly the tokens plain greedy decoding emits ("Speculative decoding changes
the speed, never the answer", splicedso primer, section "The idea"), in fewer
passes once the output repeats itself."""
import numpy as np
import pytest

import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
GREEDY = 1


def _generate(eng, batch, histories, n_tokens, gamma_max, speculate):
    """Greedy generation of n_tokens per sequence; returns (emitted streams, passes,
    per emitted token the top-2 logit margin of the row that chose it, relative to
    the logits' rms)."""
    import torch
    from speculative_decoding_verify_ragged_gb300 import draft as dr
    from workloads import device as wd
    B = batch.B
    bd = wd.batch_to_device(batch)
    lens = batch.seq_lens.astype(np.int32).copy()
    hist = [list(h) for h in histories]
    out = [[] for _ in range(B)]
    margins = [[] for _ in range(B)]
    passes = 0
    V = batch.dims["vocab"]
    while min(len(o) for o in out) < n_tokens:
        if speculate:
            dl, drafts = dr.ngram_draft_batch(hist, gamma_max, 1, 4)
        else:
            dl, drafts = np.zeros(B, np.int32), np.zeros((B, 0), np.int32)
        rows = []
        for b in range(B):
            rows.append(hist[b][-1])
            rows.extend(int(x) for x in drafts[b, :dl[b]])
        R, G = len(rows), int(dl.sum())
        bd.update(B=B, R=R, G=G, seq_lens=torch.from_numpy(lens).cuda(),
                  draft_lens=torch.from_numpy(dl.astype(np.int32)).cuda(),
                  tokens=torch.from_numpy(np.array(rows, np.int32)).cuda(), draft_probs=None, uniforms=None)
        res = wd.alloc_result(B, R, V, gamma_max, batch.page_table.shape[1], logits=True)
        eng.verify_step(bd, res)
        assert eng.read_status(res["status"]) == 0
        z = res["logits"].cpu().numpy()
        acc = res["accepted"].cpu().numpy()
        eoff = res["emitted_offsets"].cpu().numpy()
        em = res["emitted_tokens"].cpu().numpy()
        roff = np.concatenate([[0], np.cumsum(dl + 1)])
        rms = np.sqrt(np.mean(z ** 2))
        for b in range(B):
            dec = z[roff[b]: roff[b] + acc[b] + 1]             # row j chose emitted token j
            top2 = np.sort(dec, axis=1)[:, -2:]
            margins[b].extend(((top2[:, 1] - top2[:, 0]) / rms).tolist())
            toks = em[eoff[b]: eoff[b + 1]].tolist()
            out[b].extend(toks)
            hist[b].extend(toks)
        lens = res["new_seq_lens"].cpu().numpy().astype(np.int32)
        passes += 1
    return [o[:n_tokens] for o in out], passes, [m[:n_tokens] for m in margins]


def test_ngram_greedy_speculation_matches_greedy_decoding(torch_cuda_ng):
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1)
    gmax, n_tokens = 7, 96
    lens = [40, 100, 7]
    mk = lambda: wl.make_batch(wl.TINY, 71, seq_lens=lens, draft_lens=[0, 0, 0], gamma_max=gmax,  # noqa: E731
                               extra_pages=3 * (n_tokens // 16 + 2) + 6, max_pages=24)
    g = np.random.default_rng(7)
    prompts = [g.integers(0, 8, size=L + 1).tolist() for L in lens]   # the history the drafter searches
    eng = gh.engine_for(wl.TINY, gmax, wd.weights_to_device(W), 64, 8)
    eng.set_sampling(GREEDY)
    spec, p_spec, m1 = _generate(eng, mk(), prompts, n_tokens, gmax, True)
    plain, p_plain, m2 = _generate(eng, mk(), prompts, n_tokens, gmax, False)
    # the two runs sum their fp32 logits in different orders (different row counts),
    # so their argmaxes may differ only at a near-tie decision: the streams must
    # agree up to the first such decision, and at least 32 tokens in
    for b in range(len(lens)):
        for k in range(n_tokens):
            if spec[b][k] != plain[b][k]:
                assert min(m1[b][k], m2[b][k]) < 1e-4, (b, k, m1[b][k], m2[b][k])
                assert k >= 32, (b, k)
                break
    assert p_plain >= n_tokens and p_spec < p_plain


@pytest.fixture(scope="module")
def torch_cuda_ng():
    import torch
    assert torch.cuda.is_available()
    return torch
