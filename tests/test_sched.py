"""Host-side scheduler (CPU): the draft-length rule, the pages' static-versus-
continuous batching figures reproduced through the library's scheduler on the
pages' step-time line, and the slot mirror checked against the oracle's
realignment on random steps.
"""
import os

import numpy as np
import pytest

from oracle import verify_step as o

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def sched_mod():
    from speculative_decoding_verify_ragged_gb300 import _abi
    if not os.path.exists(_abi.LIB_PATH):
        from speculative_decoding_verify_ragged_gb300 import build
        build.build()
    from speculative_decoding_verify_ragged_gb300 import sched
    return sched


def _golden(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, *v = line.split()
            rows[k] = [float(x) for x in v]
    return rows


def test_draft_length_rule_matches_printed_table(sched_mod):
    for line in open(os.path.join(GOLDEN, "draft_budget.txt")):
        line = line.split("#", 1)[0].split()
        if not line:
            continue
        budget, live, per_agent = (int(x) for x in line)
        assert sched_mod.draft_length(budget, live, 1 << 20) == per_agent
    assert sched_mod.draft_length(24, 0, 8) == 0
    assert sched_mod.draft_length(24, 30, 8) == 0      # over budget: drafting off
    assert sched_mod.draft_length(512, 128, 3) == 3    # the swarm: (512 - 128) / 128
    assert sched_mod.draft_length(512, 1, 3) == 3      # capped at gamma_max


def _simulate(sched_mod, policy, lengths, floor_ms, per_seq_ms, slots=8, repeat=1):
    """Drive the scheduler with plain decoding (gamma 0) and time each step on the
    step-time line t(width) = floor + per_seq * width."""
    s = sched_mod.Scheduler(max_slots=slots, gamma_max=0, budget_rows=slots, pool_pages=1 << 20,
                            max_pages_per_seq=1 << 16, page_size=16, policy=policy)
    ids = 0
    for _ in range(repeat):
        for n in lengths:
            s.submit(ids, 0, int(n))
            ids += 1
    t_ms, steps = 0.0, []
    while True:
        st = s.plan()
        if st["live"] == 0:
            break
        assert st["gamma"] == 0 and st["rows"] == st["live"]
        t_ms += floor_ms + per_seq_ms * st["width"]
        steps.append(st)
        s.complete([0] * st["live"])
    return s.stats(), t_ms, steps


def test_static_frozen_batch_matches_printed_figures(sched_mod):
    g = _golden("static_vs_continuous.txt")
    lengths = [int(x) for x in g["lengths"]]
    st, t_ms, steps = _simulate(sched_mod, sched_mod.STATIC, lengths, g["step_ms_floor"][0], g["step_ms_per_seq"][0])
    assert st["emitted"] == sum(lengths) == g["useful_tokens"][0]
    assert st["slot_steps_paid"] == g["static_slots"][0] == len(steps) * 8
    util = 100.0 * st["slot_steps_live"] / st["slot_steps_paid"]
    assert abs(util - g["static_utilization_pct"][0]) <= g["static_utilization_pct"][1]
    tok_s = st["emitted"] / (t_ms / 1e3)
    assert abs(tok_s - g["static_tok_s"][0]) <= g["static_tok_s"][1]
    assert st["finished"] == len(lengths) and st["live"] == 0


def test_static_shrinking_batch_matches_printed_figure(sched_mod):
    g = _golden("static_vs_continuous.txt")
    lengths = [int(x) for x in g["lengths"]]
    st, t_ms, steps = _simulate(sched_mod, sched_mod.STATIC_SHRINK, lengths, g["step_ms_floor"][0],
                                g["step_ms_per_seq"][0])
    assert st["emitted"] == sum(lengths)
    assert st["slot_steps_paid"] == st["slot_steps_live"] == sum(lengths)
    # the width drops by one at each exit: 8 for the first 40 steps, ..., 1 for the last 250
    widths = [s["width"] for s in steps]
    assert widths[:40] == [8] * 40 and widths[-250:] == [1] * 250
    tok_s = st["emitted"] / (t_ms / 1e3)
    assert abs(tok_s - g["shrinking_tok_s"][0]) <= g["shrinking_tok_s"][1]


def test_continuous_batching_holds_the_full_batch(sched_mod):
    g = _golden("static_vs_continuous.txt")
    lengths = [int(x) for x in g["lengths"]]
    floor_ms, per_ms = g["step_ms_floor"][0], g["step_ms_per_seq"][0]
    st, t_ms, steps = _simulate(sched_mod, sched_mod.CONTINUOUS, lengths, floor_ms, per_ms, repeat=12)
    # while work waits every step is full: 8 tokens per t(8)
    first_short = next(i for i, s in enumerate(steps) if s["live"] < 8)
    assert first_short >= 0.75 * len(steps)
    assert all(s["live"] == 8 for s in steps[:first_short])
    # once a step runs short the queue is empty: only the drain is left
    assert all(s["admitted"] == 0 for s in steps[first_short:])
    tok_s_full = 8 / ((floor_ms + per_ms * 8) / 1e3)
    assert abs(tok_s_full - g["continuous_tok_s"][0]) <= g["continuous_tok_s"][1]
    # the whole run, drain included, beats both static policies by the pages' ~2.5x margin
    tok_s = st["emitted"] / (t_ms / 1e3)
    assert tok_s > 2.3 * g["static_tok_s"][0]
    assert st["emitted"] == 12 * sum(lengths) and st["finished"] == 12 * len(lengths)
    one = 1 / ((floor_ms + per_ms) / 1e3)
    assert abs(one - g["batch1_tok_s"][0]) <= g["batch1_tok_s"][1]


def _admit_oracle(state, ctx_lens, out_lens, gamma_max, page):
    """The oracle's admission (o.admit) on the variable-length mirror state."""
    live, n = len(state["seq_lens"]), len(ctx_lens)
    max_pages = state["page_table"].shape[1]
    pad = lambda a, fill: np.concatenate([a, np.full(n, fill, a.dtype)])  # noqa: E731
    table = dict(seq_lens=pad(state["seq_lens"], 0), num_pages=pad(state["num_pages"], 0),
                 gen_counts=pad(state["gen_counts"], 0), gen_limits=pad(state["gen_limits"], 0),
                 page_table=np.vstack([state["page_table"], np.full((n, max_pages), -1, np.int32)]))
    st, t, nf = o.admit(table, live, ctx_lens, out_lens, state["free_pages"], state["num_free"], gamma_max, page)
    assert st == o.OK
    state.update(seq_lens=t["seq_lens"], num_pages=t["num_pages"], gen_counts=t["gen_counts"],
                 gen_limits=t["gen_limits"], page_table=t["page_table"], num_free=nf)


@pytest.mark.parametrize("seed,gamma_max,budget,slots", [(0, 3, 64, 16), (1, 7, 24, 6), (2, 0, 8, 8)])
def test_mirror_follows_the_oracle_realignment(sched_mod, seed, gamma_max, budget, slots):
    """The scheduler admits what the oracle's admission rule admits, and its
    slot mirror equals the oracle's realignment + admission state after every
    step of a random run with turnover."""
    g = np.random.default_rng(seed)
    page, pool, max_pages = 16, 600, 96
    s = sched_mod.Scheduler(max_slots=slots, gamma_max=gamma_max, budget_rows=budget, pool_pages=pool,
                            max_pages_per_seq=max_pages, page_size=page)
    queue = []
    for i in range(60):
        queue.append((int(g.integers(0, 300)), int(g.integers(1, 40))))
        s.submit(i, *queue[-1])
    state = dict(seq_lens=np.zeros(0, np.int64), num_pages=np.zeros(0, np.int32),
                 page_table=np.zeros((0, max_pages), np.int32), gen_counts=np.zeros(0, np.int64),
                 gen_limits=np.zeros(0, np.int64), free_pages=g.permutation(pool).astype(np.int32), num_free=pool)
    steps = 0
    while True:
        # the scheduler admits exactly what the oracle's admission rule admits, in arrival order
        k = o.admission_count([c for c, _ in queue], len(state["seq_lens"]), state["num_free"], slots,
                              gamma_max, page)
        st = s.plan()
        assert st["admitted"] == k
        assert list(zip(st["admit_ctx"], st["admit_out"])) == queue[:k]
        queue = queue[k:]
        _admit_oracle(state, st["admit_ctx"], st["admit_out"], gamma_max, page)
        B = st["live"]
        if B == 0:
            break
        assert len(state["seq_lens"]) == B
        assert st["gamma"] == sched_mod.draft_length(budget, B, gamma_max)
        assert st["rows"] == B * (st["gamma"] + 1) and (st["gamma"] == 0 or st["rows"] <= budget)
        acc = g.integers(0, st["gamma"] + 1, size=B)
        ra = o.realign(state["seq_lens"], acc, state["page_table"], state["num_pages"], state["free_pages"],
                       state["num_free"], page, gamma_max, state["gen_counts"], state["gen_limits"])
        assert ra["status"] == o.OK
        fin = s.complete(acc)
        src = ra["next_src"]
        assert sorted(fin) == sorted(set(st["ids"]) - {st["ids"][j] for j in src})
        state.update(seq_lens=ra["next_seq_lens"].astype(np.int64), num_pages=ra["next_num_pages"],
                     page_table=ra["next_page_table"], gen_counts=ra["next_gen_counts"].astype(np.int64),
                     gen_limits=state["gen_limits"][src], free_pages=ra["free_pages"], num_free=ra["num_free"])
        m = s.slots()
        assert m["seq_lens"] == state["seq_lens"].tolist()
        assert m["gen_counts"] == state["gen_counts"].tolist()
        assert m["out_lens"] == state["gen_limits"].tolist()
        assert m["num_pages"] == state["num_pages"].tolist()
        assert s.stats()["free_pages"] == state["num_free"]
        steps += 1
    stats = s.stats()
    assert stats["finished"] == 60 and stats["queued"] == 0 and stats["free_pages"] == pool
    assert steps > 10


def test_scheduler_errors(sched_mod):
    from speculative_decoding_verify_ragged_gb300 import SdvError
    with pytest.raises(SdvError):
        sched_mod.Scheduler(max_slots=0, gamma_max=3, budget_rows=8, pool_pages=10, max_pages_per_seq=4)
    s = sched_mod.Scheduler(max_slots=2, gamma_max=3, budget_rows=8, pool_pages=10, max_pages_per_seq=4)
    with pytest.raises(SdvError):
        s.submit(0, 60, 10)          # 60 + 10 + 3 + 3 + 1 positions need 5 pages > 4
    with pytest.raises(SdvError):
        s.submit(0, 5, 0)            # an output length of zero
    s.submit(1, 5, 3)
    st = s.plan()
    assert st["live"] == 1 and st["gamma"] == 3
    with pytest.raises(SdvError):
        s.plan()                     # plan twice without completing
    with pytest.raises(SdvError):
        s.complete([4])              # more accepted than drafted
    assert s.complete([3]) == [1]    # 4 tokens >= 3: finished
    assert s.stats()["free_pages"] == 10
