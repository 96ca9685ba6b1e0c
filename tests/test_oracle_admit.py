"""Pins of the oracle's admission rule (the refill half of continuous
batching, "Why Static Batching Wastes an RX 9070 XT Agent Swarm and Continuous
Batching Wins It Back", section "Continuous batching refills the slot instead
of freezing it"): hand-worked cases, the page bookkeeping it must conserve
with the realignment, and the page's own claim that a freed slot takes a
waiting sequence on the very next step."""
import numpy as np
import pytest

from oracle import verify_step as o


def _table(slots, max_pages):
    return dict(seq_lens=np.zeros(slots, np.int64), num_pages=np.zeros(slots, np.int64),
                gen_counts=np.zeros(slots, np.int64), gen_limits=np.zeros(slots, np.int64),
                page_table=np.full((slots, max_pages), -1, np.int64))


def test_pages_for_hand_cases():
    # gamma_max 3, 16-token pages: room for the context and one block of 4 rows
    assert [o.pages_for(L, 3, 16) for L in (0, 12, 13, 15, 16, 28, 29, 100)] == [1, 1, 2, 2, 2, 2, 3, 7]
    assert o.pages_for(0, 0, 16) == 1 and o.pages_for(15, 0, 16) == 1 and o.pages_for(16, 0, 16) == 2


def test_admit_hand_case_pops_from_the_top_in_order():
    free = np.array([40, 41, 42, 43, 44, 45, 46, 47, 48, 49, 50, 51, 52, 53], np.int64)
    st, t, nf = o.admit(_table(6, 8), 0, [0, 15, 16, 60], [5, 6, 7, 8], free, 14, 3, 16)
    assert st == o.OK and nf == 14 - (1 + 2 + 2 + 4)
    assert t["num_pages"][:4].tolist() == [1, 2, 2, 4]
    assert t["page_table"][0, :2].tolist() == [53, -1]
    assert t["page_table"][1, :3].tolist() == [52, 51, -1]
    assert t["page_table"][2, :3].tolist() == [50, 49, -1]
    assert t["page_table"][3, :5].tolist() == [48, 47, 46, 45, -1]
    assert t["seq_lens"][:4].tolist() == [0, 15, 16, 60]
    assert t["gen_limits"][:4].tolist() == [5, 6, 7, 8] and t["gen_counts"][:4].tolist() == [0] * 4
    # after two survivors: their output lengths are gathered through the compaction first
    st, t2, nf2 = o.admit(t, 2, [20], [9], free, nf, 3, 16, num_live=2, next_src=[1, 3],
                          gen_limits_prev=[50, 60, 70, 80])
    assert st == o.OK and t2["gen_limits"][:3].tolist() == [60, 80, 9]
    assert t2["page_table"][2, :3].tolist() == [44, 43, -1] and nf2 == nf - 2


@pytest.mark.parametrize("case,expect", [
    (dict(live=0, ctx=[3], num_live=1), o.ERR_BAD_INPUT),      # the realignment kept 1, the host says 0
    (dict(live=0, ctx=[-1]), o.ERR_BAD_INPUT),
    (dict(live=0, ctx=[200]), o.ERR_CAPACITY),                  # 13 pages > 8 per row
    (dict(live=0, ctx=[100, 100]), o.ERR_CAPACITY),              # 14 pages > 10 free
])
def test_admit_errors_change_nothing(case, expect):
    free = np.arange(10)
    t0 = _table(4, 8)
    st, t, nf = o.admit(t0, case["live"], case["ctx"], [4] * len(case["ctx"]), free, 10, 3, 16,
                        num_live=case.get("num_live"))
    assert st == expect and nf == 10
    for k in t0:
        assert np.array_equal(t[k], t0[k])


def test_admission_count_hand_cases():
    # 10 free pages, 2 live: a 100-token newcomer needs 7 pages and leaves 3 for the growth of 3 live
    assert o.admission_count([100, 0], live=2, free_pages=10, slots=8, gamma_max=3, page=16) == 1
    # without room for the growth reserve it waits, and so does everything behind it
    assert o.admission_count([100, 0], live=3, free_pages=10, slots=8, gamma_max=3, page=16) == 0
    # slots are the other limit
    assert o.admission_count([0] * 10, live=5, free_pages=1000, slots=8, gamma_max=3, page=16) == 3
    # gamma_max 16: one step of growth is two pages per live sequence
    assert o.admission_count([0, 0], live=0, free_pages=5, slots=8, gamma_max=16, page=16) == 1


def _run(seed, slots=8, pool=400, gamma_max=3, page=16, n=60, refill=True):
    """Oracle-only continuous batching: admission, random acceptance, realignment."""
    g = np.random.default_rng(seed)
    max_pages = 64
    queue = [(int(g.integers(0, 300)), int(g.integers(1, 40))) for _ in range(n)]
    free = g.permutation(pool).astype(np.int64)
    nfree, live = pool, 0
    t = _table(slots, max_pages)
    events = []
    step = 0
    while queue or live:
        k = o.admission_count([c for c, _ in queue], live, nfree, slots, gamma_max, page) if (refill or live == 0) else 0
        adm, queue = queue[:k], queue[k:]
        st, t, nfree = o.admit(t, live, [c for c, _ in adm], [x for _, x in adm], free, nfree, gamma_max, page)
        assert st == o.OK
        live += k
        events.append((step, k, live, len(queue)))
        held = np.concatenate([t["page_table"][j, :t["num_pages"][j]] for j in range(live)] + [free[:nfree]])
        assert np.array_equal(np.sort(held), np.arange(pool))      # every page once
        if live == 0:
            break
        acc = g.integers(0, gamma_max + 1, size=live)
        ra = o.realign(t["seq_lens"][:live], acc, t["page_table"][:live], t["num_pages"][:live], free, nfree,
                       page, gamma_max, t["gen_counts"][:live], t["gen_limits"][:live])
        assert ra["status"] == o.OK
        src = ra["next_src"]
        nl = len(src)
        t2 = _table(slots, max_pages)
        t2["seq_lens"][:nl] = ra["next_seq_lens"]
        t2["num_pages"][:nl] = ra["next_num_pages"]
        t2["gen_counts"][:nl] = ra["next_gen_counts"]
        t2["gen_limits"][:nl] = t["gen_limits"][:live][src]
        t2["page_table"][:nl] = ra["next_page_table"]
        t, free, nfree, live = t2, ra["free_pages"], ra["num_free"], nl
        step += 1
    return events


def test_admission_conserves_pages_and_refills_next_step():
    events = _run(0)
    assert sum(k for _, k, _, _ in events) == 60
    # the page's claim: while work is queued (and pages are ample here), every
    # slot freed by a finished sequence is taken on the very next step
    for _, _, live, queued in events:
        if queued > 0:
            assert live == 8


def test_static_admission_leaves_slots_empty():
    """The contrast the page draws: admitting only into an empty batch leaves
    freed slots idle (fewer live slot-steps for the same work)."""
    cont = _run(1, refill=True)
    stat = _run(1, refill=False)
    assert len(stat) > len(cont)
    assert sum(e[2] for e in cont) / len(cont) > sum(e[2] for e in stat) / len(stat)
