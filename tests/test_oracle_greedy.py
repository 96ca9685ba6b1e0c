"""Greedy verification in the oracle (CPU): the emitted text equals greedy
decoding of the target, token for token, whatever the drafts ("Speculative
decoding changes the speed, never the answer", splicedso primer, section "The
idea"); the primer's token counts; ties resolved to the smallest index."""
import os

import numpy as np

from oracle import verify_step as o

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].split()
        if line:
            out.append(line)
    return out


def _markov_target(V, seed):
    """A target whose next-token distribution depends on the last token only."""
    g = np.random.default_rng(seed)
    z = g.standard_normal((V, V)) * 3
    p = np.exp(z - z.max(1, keepdims=True))
    return (p / p.sum(1, keepdims=True)).astype(np.float32)


def test_greedy_speculation_reproduces_greedy_decoding():
    V, steps = 16, 400
    P = _markov_target(V, 3)
    g = np.random.default_rng(4)
    # reference: greedy decoding, one token at a time
    ref = [5]
    for _ in range(steps + 64):
        ref.append(int(np.argmax(P[ref[-1]])))
    # speculation: drafts are right with probability 0.7 per position, random otherwise
    out = [5]
    passes = 0
    while len(out) < steps:
        gamma = int(g.integers(0, 6))
        last = out[-1]
        drafts, prev = [], last
        for _ in range(gamma):
            nxt = int(np.argmax(P[prev])) if g.random() < 0.7 else int(g.integers(0, V))
            drafts.append(nxt)
            prev = nxt
        chain = [last] + drafts                   # verify rows: the last token, then the drafts
        rows = P[np.array(chain)]                 # p at row i judges draft i + 1
        a, t = o.greedy_accept(rows, drafts)
        assert 0 <= a <= gamma
        out.extend(drafts[:a] + [t])
        passes += 1
    assert out[:steps] == ref[:steps]
    assert passes < steps                          # more than one token per pass on average


def test_greedy_primer_counts():
    V = 8
    for gamma, acc, produced in _rows("primer_example.txt"):
        gamma, acc, produced = int(gamma), int(acc), int(produced)
        rows = np.zeros((gamma + 1, V), dtype=np.float32)
        rows[np.arange(gamma + 1), 2] = 1.0        # the target always writes token 2
        drafts = [2 if i < acc else 5 for i in range(gamma)]
        a, t = o.greedy_accept(rows, drafts)
        assert a == acc and a + 1 == produced and t == 2
    # every guess right: the pass adds the target's own token after all of them
    rows = np.zeros((5, V), dtype=np.float32)
    rows[:, 2] = 1.0
    assert o.greedy_accept(rows, [2, 2, 2, 2]) == (4, 2)


def test_greedy_ties_take_the_smallest_index():
    rows = np.array([[0.1, 0.4, 0.4, 0.1], [0.3, 0.3, 0.3, 0.1]], dtype=np.float32)
    assert o.greedy_accept(rows, [2]) == (0, 1)    # 1 and 2 tie: the argmax is 1, draft 2 is rejected
    assert o.greedy_accept(rows, [1]) == (1, 0)    # accepted; the final row ties three ways -> 0


def test_greedy_batch_packs_like_stochastic():
    V = 6
    p = np.zeros((5, V), dtype=np.float32)
    p[:, 3] = 1.0
    tokens = np.array([0, 3, 3, 9 % V, 1], dtype=np.int32)   # sequence 0: last token + 2 drafts; seq 1: + 1 draft
    acc, emitted, eoff, fin = o.accept_batch(p, None, tokens, None, np.array([2, 1]), greedy=True)
    assert acc.tolist() == [2, 0] and fin.tolist() == [3, 3]
    assert eoff.tolist() == [0, 3, 4] and emitted.tolist() == [3, 3, 3, 3]
