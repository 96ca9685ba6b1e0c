"""Pins for the oracle's realignment step (CPU only).

new_len = old_len + accepted + 1 per sequence, no KV row lost or duplicated,
pages conserved between page tables and the free stack, finished sequences
release everything and survivors keep their order ("Compute Slack" post,
section "The batch also goes ragged"; "Why Static Batching Wastes an RX 9070
XT Agent Swarm", section "Continuous batching refills the slot instead of
freezing it").
"""
import numpy as np
import pytest

from oracle import verify_step as o


def _case():
    P, gmax = 4, 2
    seq_lens = [5, 10, 3]
    accepted = [1, 0, 1]
    pt = np.full((3, 6), -1, dtype=np.int32)
    pt[0, :2] = [10, 11]
    pt[1, :4] = [20, 21, 22, 23]
    pt[2, :3] = [30, 31, 32]
    npg = np.array([2, 4, 3], dtype=np.int32)
    free = np.full(16, -1, dtype=np.int32)
    free[:2] = [40, 41]
    return P, gmax, seq_lens, accepted, pt, npg, free


def test_hand_worked_case_without_finish():
    P, gmax, L, a, pt, npg, free = _case()
    r = o.realign(L, a, pt, npg, free, 2, P, gmax)
    assert r["status"] == o.OK
    assert list(r["new_seq_lens"]) == [7, 11, 5]
    # need = ceil((new_len + gmax + 1) / P) = 3, 4, 2: slot 2 gives back page 32,
    # slot 0 takes it from the top of the stack
    assert list(r["num_pages"]) == [3, 4, 2]
    assert list(r["page_table"][0, :3]) == [10, 11, 32]
    assert list(r["page_table"][2, :3]) == [30, 31, -1]
    assert r["num_free"] == 2 and list(r["free_pages"][:2]) == [40, 41]
    assert list(r["next_src"]) == [0, 1, 2]


def test_hand_worked_case_with_finish():
    P, gmax, L, a, pt, npg, free = _case()
    r = o.realign(L, a, pt, npg, free, 2, P, gmax, gen_counts=[0, 5, 0], gen_limits=[100, 6, 100])
    assert r["status"] == o.OK
    assert list(r["finished"]) == [0, 1, 0]
    assert r["num_free"] == 6
    assert list(r["free_pages"][:6]) == [40, 41, 20, 21, 22, 23]
    assert list(r["page_table"][0, :3]) == [10, 11, 32]
    assert list(r["page_table"][1]) == [-1] * 6
    assert list(r["next_src"]) == [0, 2] and r["num_live"] == 2
    assert list(r["next_seq_lens"]) == [7, 5]
    assert list(r["next_gen_counts"]) == [2, 2]


def test_capacity_error_moves_nothing():
    P, gmax, L, a, pt, npg, free = _case()
    # slot 0 needs one page, slot 2 frees one: with slot 2 over-held by zero
    # and an empty stack the pop has nothing to take
    npg2 = npg.copy()
    pt2 = pt.copy()
    pt2[2, 2] = -1
    npg2[2] = 2
    r = o.realign(L, a, pt2, npg2, free, 0, P, gmax)
    assert r["status"] == o.ERR_CAPACITY
    assert np.array_equal(r["page_table"], pt2) and np.array_equal(r["num_pages"], npg2)
    assert r["num_free"] == 0


def _random_state(g, B, P, gmax, pool):
    L = g.integers(0, 60, size=B)
    gam = g.integers(0, gmax + 1, size=B)
    a = np.array([g.integers(0, x + 1) for x in gam])
    held = (L + gmax + 1 + P - 1) // P + g.integers(0, 2, size=B)
    maxp = int(held.max()) + 4
    ids = g.permutation(pool).astype(np.int32)
    pt = np.full((B, maxp), -1, dtype=np.int32)
    o_ = 0
    for b in range(B):
        pt[b, :held[b]] = ids[o_:o_ + held[b]]
        o_ += held[b]
    free = np.full(pool, -1, dtype=np.int32)
    nfree = pool - o_
    free[:nfree] = ids[o_:]
    return L, gam, a, pt, held.astype(np.int32), free, nfree


@pytest.mark.parametrize("seed", range(25))
def test_invariants_random(seed):
    g = np.random.default_rng(seed)
    B, P, gmax = int(g.integers(1, 12)), 16 if seed % 2 else 4, int(g.integers(0, 5))
    pool = 400
    L, gam, a, pt, npg, free, nfree = _random_state(g, B, P, gmax, pool)
    gen = g.integers(0, 50, size=B)
    lim = gen + g.integers(1, 6, size=B)
    r = o.realign(L, a, pt, npg, free, nfree, P, gmax, gen_counts=gen, gen_limits=lim)
    assert r["status"] == o.OK
    new_len = np.asarray(L) + a + 1
    assert np.array_equal(r["new_seq_lens"], new_len)
    fin = (gen + a + 1) >= lim
    assert np.array_equal(r["finished"].astype(bool), fin)
    # pages conserved, none duplicated
    before = sorted(list(pt[pt >= 0]) + list(free[:nfree]))
    ptn = r["page_table"]
    after = list(ptn[ptn >= 0]) + list(r["free_pages"][:r["num_free"]])
    assert sorted(after) == before and len(set(after)) == len(after)
    for b in range(B):
        n = int(r["num_pages"][b])
        if fin[b]:
            assert n == 0
            continue
        assert n == -(-(new_len[b] + gmax + 1) // P)
        assert np.all(ptn[b, :n] >= 0) and np.all(ptn[b, n:] == -1)
        # no KV row lost: every committed position keeps its (page, slot)
        for t in range(int(new_len[b])):
            assert ptn[b, t // P] == pt[b, t // P]
    # survivors keep their order
    assert list(r["next_src"]) == [b for b in range(B) if not fin[b]]
    assert np.array_equal(r["next_page_table"], ptn[r["next_src"]])
