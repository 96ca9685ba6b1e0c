"""Continuous batching on the GPU: sdv_admit against the oracle's admission
(o.admit), and a scheduler-driven swarm whose device slot table equals, after
every step, both the oracle's realignment + admission carried on the host and
the host scheduler's mirror (through the C ABI)."""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl

pytestmark = pytest.mark.gpu


def _table(slots, max_pages):
    import torch
    z = lambda *s: torch.zeros(s, dtype=torch.int32, device="cuda")  # noqa: E731
    t = dict(seq_lens=z(slots), num_pages=z(slots), gen_counts=z(slots), gen_limits=z(slots),
             page_table=torch.full((slots, max_pages), -1, dtype=torch.int32, device="cuda"))
    return t


def _engine(gamma_max, max_rows, max_slots):
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1)
    return VerifyEngine(wd.config(wl.TINY, gamma_max), wd.weights_to_device(W), max_rows=max_rows,
                        max_slots=max_slots)


def _host(t):
    return {k: v.cpu().numpy().astype(np.int64) for k, v in t.items()}


def test_admit_matches_the_oracle():
    import torch
    gmax, page, pool, max_pages, slots = 3, 16, 64, 12, 8
    eng = _engine(gmax, 32, slots)
    g = np.random.default_rng(3)
    free = g.permutation(pool).astype(np.int32)
    t = _table(slots, max_pages)
    free_d = torch.from_numpy(free.copy()).cuda()
    nfree = torch.tensor([pool], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx = np.array([0, 15, 16, 100], np.int32)
    out = np.array([5, 6, 7, 8], np.int32)
    want_st, want, want_nf = o.admit(_host(t), 0, ctx, out, free, pool, gmax, page)
    eng.admit(t, 0, torch.from_numpy(ctx).cuda(), torch.from_numpy(out).cuda(), free_d, nfree, status)
    assert eng.read_status(status) == want_st == 0
    assert nfree.item() == want_nf
    for k, v in _host(t).items():
        assert np.array_equal(v, want[k]), k
    # a second admission after 2 survivors, gathering their limits through next_src
    prev_lim = torch.tensor([50, 60, 70, 80], dtype=torch.int32, device="cuda")
    t["gen_limits"].zero_()
    before = _host(t)
    src = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    nlive = torch.tensor([2], dtype=torch.int32, device="cuda")
    want_st, want, want_nf = o.admit(before, 2, [30], [9], free, nfree.item(), gmax, page, num_live=2,
                                     next_src=[1, 3], gen_limits_prev=[50, 60, 70, 80])
    eng.admit(t, 2, torch.tensor([30], dtype=torch.int32, device="cuda"),
              torch.tensor([9], dtype=torch.int32, device="cuda"), free_d, nfree, status,
              num_live=nlive, next_src=src, gen_limits_prev=prev_lim)
    assert eng.read_status(status) == want_st == 0
    assert nfree.item() == want_nf
    for k, v in _host(t).items():
        assert np.array_equal(v, want[k]), k


def test_admit_device_errors_write_nothing():
    import torch
    eng = _engine(3, 16, 4)
    t = _table(4, 8)
    free_d = torch.arange(10, dtype=torch.int32, device="cuda")
    nfree = torch.tensor([10], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # 200 positions need 13 pages > 8 per row and > 10 free
    eng.admit(t, 0, torch.tensor([200], dtype=torch.int32, device="cuda"),
              torch.tensor([4], dtype=torch.int32, device="cuda"), free_d, nfree, status)
    assert eng.read_status(status) == 2   # SDV_ERR_CAPACITY
    assert nfree.item() == 10 and int((t["page_table"] >= 0).sum().item()) == 0
    status.zero_()
    nlive = torch.tensor([1], dtype=torch.int32, device="cuda")
    eng.admit(t, 0, torch.tensor([3], dtype=torch.int32, device="cuda"),
              torch.tensor([4], dtype=torch.int32, device="cuda"), free_d, nfree, status, num_live=nlive)
    assert eng.read_status(status) == 6   # SDV_ERR_BAD_INPUT: the realignment kept 1, the host says 0
    assert nfree.item() == 10
    status.fill_(5)                       # an earlier failure: a no-op
    eng.admit(t, 0, torch.tensor([3], dtype=torch.int32, device="cuda"),
              torch.tensor([4], dtype=torch.int32, device="cuda"), free_d, nfree, status)
    assert nfree.item() == 10


def _random_drafter(V, key):
    import torch
    from workloads import device as wd

    def fill(st, batch):
        k = key + 1000 * fill.n
        fill.n += 1
        g = wl.rng(9, wl.S_TOKENS, k)
        batch["tokens"] = torch.from_numpy(g.integers(0, V, size=st["rows"]).astype(np.int32)).cuda()
        batch["draft_probs"] = wd.draft_probs_device(st["drafts"], V, wl._key(9, wl.S_Q, k))
        batch["uniforms"] = torch.from_numpy(wl.uniform24(wl.rng(9, wl.S_U, k), st["rows"])).cuda()
    fill.n = 0
    return fill


@pytest.mark.parametrize("budget,slots", [(24, 6), (12, 8)])
def test_swarm_runner_device_table_equals_the_scheduler_mirror(budget, slots):
    import torch
    from speculative_decoding_verify_ragged_gb300.serve import SwarmRunner
    from workloads import device as wd
    gmax, page, pool_pages, max_pages = 3, 16, 160, 40
    d = wl.TINY
    eng = _engine(gmax, slots * (gmax + 1), slots)
    pool = torch.empty((pool_pages, d["n_kv"], 2, page, d["head_dim"]), dtype=torch.bfloat16, device="cuda")
    wd.normal_bf16_device_(pool, wl._key(9, wl.S_KV, 0))
    run = SwarmRunner(eng, pool, pool_pages, slots, budget, max_pages)
    g = np.random.default_rng(budget)
    outs, queue, admitted = [], [], 0
    for i in range(24):
        outs.append(int(g.integers(2, 30)))
        queue.append((int(g.integers(0, 200)), outs[-1]))
        run.submit(i, queue[-1][0], outs[-1])
    drafter = _random_drafter(d["vocab"], budget)
    # the oracle's state: admission and realignment carried on the host from
    # the scheduler's plans and the GPU's accepted counts
    ot = _host(_table(slots, max_pages))
    ofree, onf, olive = np.arange(pool_pages, dtype=np.int64), pool_pages, 0
    steps = 0
    while True:
        st, batch = run.plan()
        if st["live"] == 0:
            break
        assert st["admitted"] == o.admission_count(
            [c for c, _ in queue[admitted:]], olive, onf, slots, gmax, page)
        code, ot, onf = o.admit(ot, olive, st["admit_ctx"], st["admit_out"], ofree, onf, gmax, page)
        assert code == o.OK
        admitted += st["admitted"]
        olive += st["admitted"]
        assert np.array_equal(_host(run.table())["page_table"][:olive], ot["page_table"][:olive])
        drafter(st, batch)
        run.verify(st, batch)
        fin = run.complete(st)
        acc = run.res["accepted"][:olive].cpu().numpy()
        ra = o.realign(ot["seq_lens"][:olive], acc, ot["page_table"][:olive], ot["num_pages"][:olive], ofree,
                       onf, page, gmax, ot["gen_counts"][:olive], ot["gen_limits"][:olive])
        assert ra["status"] == o.OK
        src, nl = ra["next_src"], ra["num_live"]
        nt = _host(_table(slots, max_pages))
        nt["seq_lens"][:nl], nt["num_pages"][:nl] = ra["next_seq_lens"], ra["next_num_pages"]
        nt["gen_counts"][:nl], nt["page_table"][:nl] = ra["next_gen_counts"], ra["next_page_table"]
        nt["gen_limits"][:nl] = ot["gen_limits"][:olive][src]
        ot, ofree, onf, olive = nt, ra["free_pages"].astype(np.int64), ra["num_free"], nl
        steps += 1
        assert st["rows"] == st["live"] * (st["gamma"] + 1)
        m = run.sched.slots()
        n = len(m["seq_lens"])
        assert n == olive
        t = run.table()
        # the device table against the oracle (the limits are gathered at the next admission)
        for k in ("seq_lens", "gen_counts", "num_pages", "page_table"):
            assert np.array_equal(_host(t)[k][:n], ot[k][:n]), k
        assert run.num_free.item() == onf
        assert np.array_equal(run.free_pages[:onf].cpu().numpy(), ofree[:onf])
        # and against the scheduler's own mirror
        assert t["seq_lens"][:n].cpu().tolist() == m["seq_lens"]
        assert t["gen_counts"][:n].cpu().tolist() == m["gen_counts"]
        assert t["num_pages"][:n].cpu().tolist() == m["num_pages"]
        assert run.num_free.item() == run.sched.stats()["free_pages"]
        # every pool page held by one live slot or free, once
        pt = t["page_table"][:n].cpu().numpy()
        held = np.concatenate([pt[j, :m["num_pages"][j]] for j in range(n)] +
                              [run.free_pages[:run.num_free.item()].cpu().numpy()])
        assert np.array_equal(np.sort(held), np.arange(pool_pages))
    s = run.sched.stats()
    assert s["finished"] == 24 and s["free_pages"] == pool_pages and steps > 5
    # the output limits carried through the compactions: every sequence stopped at its own
    # length, overshooting by at most the drafts of its last step
    assert sum(outs) <= s["emitted"] <= sum(outs) + 24 * gmax
