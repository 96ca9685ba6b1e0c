"""Token trees on the GPU (greedy verification, through the C ABI) against the
oracle: "a small tree" of drafts per sequence ("Speculative Decoding and
Batching Compete for the Same Compute Slack on RDNA4", table in "What the
budget says to build").  Each node attends to the cache and its own ancestors
at rotary position L + depth, acceptance walks down the argmax matches, and the
accepted path's K/V rows move to consecutive cache slots."""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
GREEDY, STOCHASTIC = 1, 0
BAD_INPUT, UNSUPPORTED = 6, 7


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available()
    return torch


def _random_tree(g, n):
    """n nodes; node c hangs under a uniformly chosen earlier node."""
    return [-1] + [int(g.integers(0, c)) for c in range(1, n)]


def _tree_batch(dims, trees, lens, seed, gmax):
    gam = [len(t) - 1 for t in trees]
    b = wl.make_batch(dims, 300 + seed, seq_lens=lens, draft_lens=gam, gamma_max=gmax, extra_pages=2 * len(lens) + 4)
    parents = np.concatenate([np.array(t, dtype=np.int32) for t in trees])
    return b, parents


def _plant(batch, W, trees, parents, g):
    """Set chosen nodes' tokens to their parent's argmax (in depth order, one
    oracle forward per depth): along one root-to-leaf path per tree (the first
    tree's deepest, a random one elsewhere, sometimes cut short), and at a later
    sibling of a planted node with the same token, so that the walk's
    smallest-index rule decides."""
    roff = wl.row_offsets(batch.draft_lens)
    plan = []  # (row, parent row, depth)
    for s, t in enumerate(trees):
        depth = o.tree_depths(t)
        leaves = [v for v in range(len(t)) if v not in t[1:]]
        leaf = max(leaves, key=lambda v: depth[v]) if s == 0 else leaves[int(g.integers(0, len(leaves)))]
        path = o.tree_ancestors(t, leaf)[1:]
        # stop the planted path early in some trees
        if s > 0 and path and g.random() < 0.4:
            path = path[:int(g.integers(0, len(path)))]
        for v in path:
            plan.append((int(roff[s]) + v, int(roff[s]) + t[v], depth[v]))
            twins = [c for c in range(v + 1, len(t)) if t[c] == t[v]]
            if twins and g.random() < 0.5:
                plan.append((int(roff[s]) + twins[0], int(roff[s]) + t[v], depth[v]))
    for d in range(1, max([p[2] for p in plan], default=0) + 1):
        fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens,
                       batch.tokens, parents=parents)
        for r, pr, dep in plan:
            if dep == d:
                batch.tokens[r] = int(np.argmax(fw["logits"][pr]))


def _run(eng, batch, parents):
    import torch
    from workloads import device as wd
    bd = wd.batch_to_device(batch)
    bd["tree_parents"] = torch.from_numpy(parents).cuda()
    bd["draft_probs"] = None
    bd["uniforms"] = None
    pt_before = batch.page_table.copy()
    res = wd.alloc_result(batch.B, batch.R, batch.dims["vocab"], batch.gamma_max, batch.page_table.shape[1],
                          logits=True)
    eng.verify_step(bd, res)
    status = eng.read_status(res["status"])
    torch.cuda.synchronize()
    return status, gh.to_numpy(res), gh.to_numpy(bd), pt_before


def _final_nodes(batch, trees, paths):
    """Which node's K/V each slot L + j holds after compaction: o.compact_kv run
    on a pool of node labels."""
    P = batch.dims["page"]
    pages = batch.kv_pool.shape[0]
    lab = np.zeros((pages, 1, 1, P, 1), dtype=np.int64) - 1
    for s, t in enumerate(trees):
        L = int(batch.seq_lens[s])
        for v in range(len(t)):
            pos = L + v
            lab[batch.page_table[s, pos // P], 0, 0, pos % P, 0] = v
    moved = o.compact_kv(lab, batch.page_table, batch.seq_lens, paths, P)
    out = {}
    for s, t in enumerate(trees):
        L = int(batch.seq_lens[s])
        for v in range(len(t)):
            pos = L + v
            out[(s, pos)] = int(moved[batch.page_table[s, pos // P], 0, 0, pos % P, 0])
    return out


def _paths_from_emitted(batch, trees, res):
    """Each sequence's accepted path (node indices at depths 1..a) from the
    GPU's emitted tokens: at each depth, the smallest-index child of the current
    node whose token is the emitted one."""
    eoff = res["emitted_offsets"]
    roff = wl.row_offsets(batch.draft_lens)
    paths = []
    for s, t in enumerate(trees):
        node_tok = batch.tokens[int(roff[s]): int(roff[s]) + len(t)]
        toks = res["emitted_tokens"][eoff[s]: eoff[s + 1]]
        a = int(res["accepted"][s])
        v, path = 0, []
        for k in range(a):
            kids = [c for c in range(1, len(t)) if t[c] == v and int(node_tok[c]) == int(toks[k])]
            assert kids, (s, k, "no child carries the emitted token")
            v = kids[0]
            path.append(v)
        paths.append(path)
    return paths


def _check_tree_step(eng, W, batch, trees, parents, name):
    status, res, dev, pt_before = _run(eng, batch, parents)
    assert status == 0, f"{name}: status {status}"
    ref = o.verify_step(batch, W, greedy=True, parents=parents)
    fw = ref["forward"]
    z = ref["logits"]
    tol = gh.LOGIT_TOL_REL_RMS * np.sqrt(np.mean(z ** 2))
    assert np.abs(res["logits"] - z).max() <= tol, name
    top2 = np.sort(z, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 2 * tol
    roff = wl.row_offsets(batch.draft_lens)
    same = np.ones(batch.B, dtype=bool)
    for s in range(batch.B):
        # the rows the oracle's walk decided at: the root and every node of its path
        visited = [0] + list(ref["paths"][s])
        if not all(clear[int(roff[s]) + v] for v in visited):
            same[s] = False
            continue
        assert int(res["accepted"][s]) == int(ref["accepted"][s]), (name, s)
        assert int(res["final_tokens"][s]) == int(ref["final_tokens"][s]), (name, s)
    assert same.sum() >= batch.B // 2, (name, same)
    assert np.array_equal(res["new_seq_lens"], batch.seq_lens + res["accepted"] + 1)
    # realignment and the cache moves are checked from the GPU's own walk, always:
    # its path is recovered from its emitted tokens (at each depth the smallest
    # child of the current node carrying the emitted token, the walk's rule)
    paths = _paths_from_emitted(batch, trees, res)
    for s, t in enumerate(trees):
        if same[s]:
            assert paths[s] == list(ref["paths"][s]), (name, s)
        # every slot: each choice of the GPU's walk (the tokens it descended by and
        # its final token) is within the logit tolerance of the oracle's maximum at
        # the row it was taken at, and the walk stopped where no child carries its
        # final token
        r0 = int(roff[s])
        visited = [0] + paths[s]
        chosen = [int(batch.tokens[r0 + v]) for v in paths[s]] + [int(res["final_tokens"][s])]
        for v, tok in zip(visited, chosen):
            assert z[r0 + v, tok] >= z[r0 + v].max() - 2 * tol, (name, s, v, tok)
        assert not any(t[c] == visited[-1] and int(batch.tokens[r0 + c]) == chosen[-1] for c in range(1, len(t)))
    ra = o.realign(batch.seq_lens, res["accepted"], batch.page_table, batch.num_pages, batch.free_pages,
                   batch.num_free, batch.dims["page"], batch.gamma_max)
    eoff = np.concatenate([[0], np.cumsum(res["accepted"].astype(np.int64) + 1)])
    assert np.array_equal(res["emitted_offsets"], eoff)
    for s, t in enumerate(trees):
        toks = [int(batch.tokens[int(roff[s]) + v]) for v in paths[s]] + [int(res["final_tokens"][s])]
        assert res["emitted_tokens"][eoff[s]: eoff[s + 1]].tolist() == toks, (name, s)
    assert np.array_equal(dev["page_table"], ra["page_table"])
    nf = int(dev["num_free_out"][0])
    assert nf == ra["num_free"] and np.array_equal(dev["free_pages"][:nf], ra["free_pages"][:nf])
    # the cache: every verified slot holds the K/V of the node compaction puts
    # there (a bf16 rounding within the window of the oracle's value);
    # every other slot of the pool is untouched
    where = _final_nodes(batch, trees, paths)
    pool = dev["kv_pool"].view(np.uint16) if dev["kv_pool"].dtype != np.uint16 else dev["kv_pool"]
    P = batch.dims["page"]
    local = {int(r): n for n, r in enumerate(fw["rows"])}
    touched = np.zeros(pool.shape[:1] + pool.shape[3:4], dtype=bool)  # [page, slot]
    for (s, pos), v in where.items():
        n = local[int(roff[s]) + v]
        pg = pt_before[s, pos // P]
        touched[pg, pos % P] = True
        for kind, kv in (("k", 0), ("v", 1)):
            got = o.bf16_to_f64(pool[pg, :, kv, pos % P, :])
            pre = fw[kind + "_pre"][n]
            e_ = gh.KV_WINDOW * np.sqrt(np.mean(pre ** 2, axis=1, keepdims=True))
            ok = (o.round_bf16(pre - e_) <= got) & (got <= o.round_bf16(pre + e_))
            assert ok.all(), (name, kind, s, pos, v)
    rest = ~touched
    assert np.array_equal(pool.transpose(0, 3, 1, 2, 4)[rest], batch.kv_pool.transpose(0, 3, 1, 2, 4)[rest])
    return ref


def test_tree_step_tiny(torch_cuda):
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1)
    gmax = 15
    eng = gh.engine_for(wl.TINY, gmax, wd.weights_to_device(W), 128, 16)
    eng.set_sampling(GREEDY)
    g = np.random.default_rng(5)
    trees = [[-1], [-1, 0, 1, 2], [-1, 0, 0, 0, 0], _random_tree(g, 16), _random_tree(g, 9),
             [-1, 0, 0, 1, 1, 2, 3, 0, 5], _random_tree(g, 12), _random_tree(g, 3)]
    lens = [40, 0, 15, 200, 31, 77, 129, 16]
    batch, par = _tree_batch(wl.TINY, trees, lens, 1, gmax)
    _plant(batch, W, trees, par, g)
    ref = _check_tree_step(eng, W, batch, trees, par, "tiny-tree")
    assert int(ref["accepted"].max()) >= 3


@pytest.mark.parametrize("path", [1, 2])
def test_tree_step_nine_b(torch_cuda, nine_b_weights, path):
    """The 9B-class layer: both attention kernels, trees of up to 8 nodes (32
    query vectors per KV head at 4 query heads per KV head)."""
    W, Wd = nine_b_weights
    gmax = 7
    eng = gh.engine_for(wl.NINE_B, gmax, Wd, 64, 8)
    eng.set_sampling(GREEDY)
    eng.set_attention_path(path)
    g = np.random.default_rng(6 + path)
    trees = [_random_tree(g, 8), [-1, 0, 0, 1, 2, 1, 0, 3], [-1, 0], _random_tree(g, 6), [-1]]
    lens = [2048, 513, 1000, 15, 64]
    batch, par = _tree_batch(wl.NINE_B, trees, lens, 2 + path, gmax)
    _plant(batch, W, trees, par, g)
    ref = _check_tree_step(eng, W, batch, trees, par, f"nine-b-tree-{path}")
    assert int(ref["accepted"].max()) >= 2


def test_tree_step_nine_b_sixteen_nodes(torch_cuda, nine_b_weights):
    """The tree size the pages name for one agent, ~8 to 16 deep ("Speculative
    Decoding and Batching Compete for the Same Compute Slack on RDNA4", table
    in "What the budget says to build"): 16-node trees on the 9B-class layer,
    64 query vectors per KV head, which the tcgen05 attention kernel takes in
    two items of 32."""
    W, Wd = nine_b_weights
    gmax = 15
    eng = gh.engine_for(wl.NINE_B, gmax, Wd, 64, 8)
    eng.set_sampling(GREEDY)
    eng.set_attention_path(2)
    g = np.random.default_rng(16)
    chain16 = list(range(-1, 15))
    trees = [_random_tree(g, 16), chain16, [-1] + [0] * 15, _random_tree(g, 11)]
    lens = [2048, 700, 3000, 31]
    batch, par = _tree_batch(wl.NINE_B, trees, lens, 16, gmax)
    _plant(batch, W, trees, par, g)
    ref = _check_tree_step(eng, W, batch, trees, par, "nine-b-tree-16")
    assert int(ref["accepted"].max()) >= 3


@pytest.mark.parametrize("path", [1, 2])
def test_chain_shaped_tree_equals_chain(torch_cuda, nine_b_weights, path):
    """A tree whose every node hangs under the one before is the chain: the same
    logits to the bit, the same acceptance, the same cache."""
    import torch
    from workloads import device as wd
    W, Wd = nine_b_weights
    gmax = 7
    eng = gh.engine_for(wl.NINE_B, gmax, Wd, 64, 8)
    eng.set_sampling(GREEDY)
    eng.set_attention_path(path)
    lens, gam = [300, 17, 4000, 0, 64], [7, 3, 0, 5, 2]
    outs = []
    for tree in (False, True):
        batch = wl.make_batch(wl.NINE_B, 330, seq_lens=lens, draft_lens=gam, gamma_max=gmax, extra_pages=12)
        bd = wd.batch_to_device(batch)
        if tree:
            bd["tree_parents"] = torch.from_numpy(
                np.concatenate([np.arange(-1, g_, dtype=np.int32) for g_ in gam])).cuda()
        res = wd.alloc_result(batch.B, batch.R, wl.NINE_B["vocab"], gmax, batch.page_table.shape[1], logits=True)
        eng.verify_step(bd, res)
        assert eng.read_status(res["status"]) == 0
        outs.append((gh.to_numpy(res), gh.to_numpy(bd)))
    (r0, d0), (r1, d1) = outs
    assert np.array_equal(r0["logits"], r1["logits"])
    for k in ("accepted", "final_tokens", "emitted_offsets", "emitted_tokens", "new_seq_lens"):
        assert np.array_equal(r0[k], r1[k]), k
    assert np.array_equal(d0["kv_pool"], d1["kv_pool"])
    assert np.array_equal(d0["page_table"], d1["page_table"])


@pytest.mark.parametrize("gmax", [7, 11])
def test_tree_attention_matches_oracle(torch_cuda, gmax):
    """Attention alone (sdv_attention, both kernels) on a 9B-shaped batch of
    trees: node i's query sees the cache and its ancestors' keys only.  Trees
    of up to 8 nodes fill the tcgen05 kernel's 32-vector items, up to 12 its
    48-vector items."""
    torch = torch_cuda
    from workloads import device as wd
    from tests.test_gpu_parity import _attn_only_engine
    dims = wl.NINE_B
    g = np.random.default_rng(9 + gmax)
    trees = [_random_tree(g, int(g.integers(1, gmax + 2))) for _ in range(12)]
    trees[0] = _random_tree(g, gmax + 1)
    lens = [int(x) for x in g.integers(0, 2500, size=12)]
    b, par = _tree_batch(dims, trees, lens, 9, gmax)
    R, nq, nkv, D, P = b.R, dims["n_q"], dims["n_kv"], dims["head_dim"], dims["page"]
    q = g.standard_normal((R, nq, D)).astype(np.float32)
    pool = o.bf16_to_f64(b.kv_pool)
    offs = wl.row_offsets(b.draft_lens)
    ref = np.zeros((R, nq * D))
    for s, t in enumerate(trees):
        L = int(b.seq_lens[s])
        Kc, Vc = o.gather_kv(pool, b.page_table[s], L + len(t), P)
        for i in range(len(t)):
            keys = list(range(L)) + [L + j for j in o.tree_ancestors(t, i)]
            r = int(offs[s]) + i
            for h in range(nq):
                kv = h // (nq // nkv)
                ref[r, h * D:(h + 1) * D] = o.attention_one(q[r, h].astype(np.float64), Kc[kv, keys], Vc[kv, keys])
    eng = _attn_only_engine(wd.config(dims, gmax), torch)
    rms = np.sqrt(np.mean(ref ** 2))
    for path in (1, 2):
        eng.set_attention_path(path)
        bd = wd.batch_to_device(b)
        bd["tree_parents"] = torch.from_numpy(par).cuda()
        out = torch.zeros((R, nq * D), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        eng.attention(torch.from_numpy(q).cuda(), bd, out, st)
        assert eng.read_status(st) == 0
        err = np.abs(out.cpu().numpy() - ref)
        assert err.max() <= 1e-3 * rms + 1e-4 * np.abs(ref).max(), (path, err.max(), rms)


def test_tree_errors(torch_cuda):
    """Trees with stochastic sampling, a realignment without the path, and
    malformed parent tables are refused (host) or reported (device status)."""
    import torch
    from speculative_decoding_verify_ragged_gb300 import SdvError
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1)
    eng = gh.engine_for(wl.TINY, 4, wd.weights_to_device(W), 64, 8)
    trees = [[-1, 0, 0], [-1, 0, 1, 1]]
    batch, par = _tree_batch(wl.TINY, trees, [10, 20], 4, 4)
    bd = wd.batch_to_device(batch)
    bd["tree_parents"] = torch.from_numpy(par).cuda()
    res = wd.alloc_result(batch.B, batch.R, wl.TINY["vocab"], 4, batch.page_table.shape[1])
    eng.set_sampling(STOCHASTIC)
    with pytest.raises(SdvError) as ei:
        eng.verify_step(bd, res)
    assert ei.value.code == UNSUPPORTED
    eng.set_sampling(GREEDY)
    with pytest.raises(SdvError) as ei:
        eng.realign(bd, res)
    assert ei.value.code == UNSUPPORTED
    for bad in ([0, 0, 0, -1, 0, 1, 1], [-1, 0, 2, -1, 0, 1, 1], [-1, 0, 0, -1, 0, 1, 3], [-1, 0, 0, -1, -1, 1, 1]):
        b2 = wl.make_batch(wl.TINY, 304, seq_lens=[10, 20], draft_lens=[2, 3], gamma_max=4, extra_pages=8)
        bd = wd.batch_to_device(b2)
        bd["tree_parents"] = torch.tensor(bad, dtype=torch.int32, device="cuda")
        bd["draft_probs"] = None
        bd["uniforms"] = None
        res = wd.alloc_result(b2.B, b2.R, wl.TINY["vocab"], 4, b2.page_table.shape[1])
        eng.verify_step(bd, res)
        assert eng.read_status(res["status"]) == BAD_INPUT, bad
        # nothing moved: the page tables are as they were
        assert np.array_equal(bd["page_table"].cpu().numpy(), b2.page_table)


@pytest.mark.parametrize("dims,B,seed", [(wl.TINY, 12, 0), (wl.NINE_B, 10, 1), (wl.TINY, 40, 2)])
def test_tree_accept_bit_exact(torch_cuda, dims, B, seed):
    """Acceptance and realignment on given probabilities (sdv_accept): the walk,
    the emitted path, the page tables and the moved cache rows equal the
    oracle's to the bit (o.compact_kv on the pool as it was)."""
    import torch
    from workloads import device as wd
    g = np.random.default_rng(40 + seed)
    V = dims["vocab"]
    gmax = 7 if dims is wl.NINE_B else 15
    trees = [_random_tree(g, int(g.integers(1, gmax + 2))) for _ in range(B)]
    lens = [int(x) for x in g.integers(0, 400, size=B)]
    b, par = _tree_batch(dims, trees, lens, 20 + seed, gmax)
    p = wl.softmax_f32(g.standard_normal((b.R, V)).astype(np.float32) * 2)
    roff = wl.row_offsets(b.draft_lens)
    for s, t in enumerate(trees):
        # nodes take their parent's argmax with probability 0.8 (twins make ties)
        for c in range(1, len(t)):
            if g.random() < 0.8:
                b.tokens[int(roff[s]) + c] = int(np.argmax(p[int(roff[s]) + t[c]]))
    if dims is wl.NINE_B:
        from tests.test_gpu_parity import _attn_only_engine
        eng = _attn_only_engine(wd.config(dims, gmax), torch)
    else:
        eng = gh.engine_for(dims, gmax, wd.weights_to_device(wl.make_weights(wl.TINY, 1)), max(b.R, 16), 64)
    eng.set_sampling(GREEDY)
    bd = wd.batch_to_device(b)
    bd["tree_parents"] = torch.from_numpy(par).cuda()
    bd["draft_probs"] = None
    bd["uniforms"] = None
    res = wd.alloc_result(b.B, b.R, V, gmax, b.page_table.shape[1])
    eng.accept(torch.from_numpy(p).cuda(), bd, res)
    assert eng.read_status(res["status"]) == 0
    acc, emitted, eoff, fin, paths = o.accept_batch(p, None, b.tokens, None, b.draft_lens, greedy=True, parents=par)
    r = gh.to_numpy(res)
    d = gh.to_numpy(bd)
    assert np.array_equal(r["accepted"], acc)
    assert np.array_equal(r["final_tokens"], fin)
    assert np.array_equal(r["emitted_offsets"], eoff)
    assert np.array_equal(r["emitted_tokens"][:eoff[-1]], emitted)
    ra = o.realign(b.seq_lens, acc, b.page_table, b.num_pages, b.free_pages, b.num_free, dims["page"], gmax)
    assert np.array_equal(d["page_table"], ra["page_table"])
    want = o.compact_kv(b.kv_pool, b.page_table, b.seq_lens, paths, dims["page"])
    assert np.array_equal(d["kv_pool"], want)
    assert acc.max() >= 2 and any(len(pth) and pth != list(range(1, len(pth) + 1)) for pth in paths)
