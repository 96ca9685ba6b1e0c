"""Token trees in the oracle (CPU): a chain-shaped tree is the chain; every node
of a branching tree computes what the chain of its own root-to-node path
computes (attention to its ancestors only, rotary position = depth); greedy
verification of trees emits the target's greedy chain; the accepted path's K/V
rows move to consecutive slots."""
import numpy as np

from oracle import verify_step as o
import workloads as wl


def _tree_batch(parents_per_seq, lens, seed):
    gam = [len(p) - 1 for p in parents_per_seq]
    b = wl.make_batch(wl.TINY, 80 + seed, seq_lens=lens, draft_lens=gam, gamma_max=max(gam), extra_pages=4)
    parents = np.concatenate([np.array(p, dtype=np.int32) for p in parents_per_seq])
    return b, parents


def test_chain_shaped_tree_is_the_chain():
    W = wl.make_weights(wl.TINY, 1)
    b, par = _tree_batch([[-1, 0, 1, 2], [-1, 0]], [20, 5], 0)
    f0 = o.forward(b.dims, W, b.kv_pool, b.page_table, b.seq_lens, b.draft_lens, b.tokens)
    f1 = o.forward(b.dims, W, b.kv_pool, b.page_table, b.seq_lens, b.draft_lens, b.tokens, parents=par)
    assert np.array_equal(f0["logits"], f1["logits"])


def test_every_node_computes_its_own_path():
    W = wl.make_weights(wl.TINY, 1)
    tree = [-1, 0, 0, 1, 1, 2, 3, 0, 5]     # root 0; children 1, 2, 7; 3, 4 under 1; 5 under 2; 6 under 3; 8 under 5
    L = 24
    b, par = _tree_batch([tree], [L], 1)
    ft = o.forward(b.dims, W, b.kv_pool, b.page_table, b.seq_lens, b.draft_lens, b.tokens, parents=par)
    z = ft["logits"]
    rms = np.sqrt(np.mean(z ** 2))
    for v in range(len(tree)):
        path = o.tree_ancestors(tree, v)                      # root .. v in order (indices increase along a path)
        chain = wl.make_batch(wl.TINY, 80 + 1, seq_lens=[L], draft_lens=[len(path) - 1], gamma_max=len(tree),
                              extra_pages=4)
        chain.kv_pool = b.kv_pool.copy()
        chain.page_table = b.page_table.copy()
        chain.tokens = b.tokens[np.array(path)]
        fc = o.forward(chain.dims, W, chain.kv_pool, chain.page_table, chain.seq_lens, chain.draft_lens,
                       chain.tokens)
        assert np.abs(fc["logits"][len(path) - 1] - z[v]).max() <= 1e-9 * rms, v
    # the K/V of node v is written at slot L + v, rotated for position L + depth(v)
    depth = o.tree_depths(tree)
    assert sorted(ft["kv_rows"].keys()) == [(0, L + v) for v in range(len(tree))]
    assert depth == [0, 1, 1, 2, 2, 2, 3, 1, 3]


def _markov(V, seed):
    g = np.random.default_rng(seed)
    z = g.standard_normal((V, V)) * 3
    p = np.exp(z - z.max(1, keepdims=True))
    return p / p.sum(1, keepdims=True)


def test_greedy_tree_speculation_reproduces_greedy_decoding():
    V, n = 12, 300
    P = _markov(V, 2)
    g = np.random.default_rng(3)
    ref = [4]
    for _ in range(n + 40):
        ref.append(int(np.argmax(P[ref[-1]])))
    out, passes = [4], 0
    while len(out) < n:
        # a random tree of up to 12 nodes; each new node hangs under a random earlier node and
        # guesses the target's next token with probability 0.5
        tokens, parents = [out[-1]], [-1]
        for c in range(1, int(g.integers(1, 13))):
            par = int(g.integers(0, c))
            guess = int(np.argmax(P[tokens[par]])) if g.random() < 0.5 else int(g.integers(0, V))
            tokens.append(guess)
            parents.append(par)
        rows = P[np.array(tokens)]                  # node v's row: the target after node v's token
        a, t, path = o.greedy_tree_accept(rows, tokens, parents)
        assert len(path) == a and (not path or parents[path[0]] == 0)
        for k in range(1, a):
            assert parents[path[k]] == path[k - 1]
        out.extend([tokens[c] for c in path] + [t])
        passes += 1
    assert out[:n] == ref[:n]
    assert passes < n * 0.8


def test_greedy_tree_walk_hand_cases():
    V = 5
    rows = np.zeros((6, V))
    # node tokens: root 9 (ignored), 1: 2, 2: 3, 3: 3, 4: 1, 5: 0
    tokens = [9, 2, 3, 3, 1, 0]
    parents = [-1, 0, 0, 0, 2, 4]
    rows[0, 3] = 1        # the root wants 3: children 2 and 3 both carry 3 -> the smaller index, 2
    rows[2, 1] = 1        # node 2 wants 1: child 4
    rows[4, 4] = 1        # node 4 wants 4: child 5 carries 0 -> stop at node 4, final token 4
    assert o.greedy_tree_accept(rows, tokens, parents) == (2, 4, [2, 4])
    rows[0] = 0
    rows[0, 4] = 1        # nothing under the root carries 4: no draft kept
    assert o.greedy_tree_accept(rows, tokens, parents) == (0, 4, [])


def test_compact_kv_moves_the_path_rows():
    P = 4
    pool = np.arange(6 * 1 * 2 * P * 2, dtype=np.uint16).reshape(6, 1, 2, P, 2)
    page_table = np.array([[3, 1, 5, -1]], dtype=np.int32)
    L = 2
    out = o.compact_kv(pool, page_table, [L], [[3, 5]], P)
    # depth 1 <- node 3: slot 3 (page 3, row 3) <- slot 5 (page 1, row 1)
    assert np.array_equal(out[3, :, :, 3], pool[1, :, :, 1])
    # depth 2 <- node 5: slot 4 (page 1, row 0) <- slot 7 (page 1, row 3)
    assert np.array_equal(out[1, :, :, 0], pool[1, :, :, 3])
    untouched = np.ones(pool.shape, dtype=bool)
    untouched[3, :, :, 3] = False
    untouched[1, :, :, 0] = False
    assert np.array_equal(out[untouched], pool[untouched])
