"""Continuous-batching swarm drivers for the tests (test infrastructure).

The swarm follows the pages' agent-swarm loop: B slots verify drafts every
step; a sequence finishes when its emitted count reaches its output length
(log-uniform), its slot is removed by stable compaction and refilled with a
new sequence (fresh context length, synthetic KV, no prefill); every slot
drafts gamma = clamp((budget - B_live) / B_live, 0, gamma_max) tokens.

Two drivers:

* ``OracleSwarm`` carries the state the oracle computes (KV cache with the
  oracle's own K/V rows, lengths, pages, free stack).  Each step's inputs come
  from that state and the seeded generators only, so the GPU is compared with
  the oracle at every step without ever feeding a GPU result back in.
* ``DeviceSwarm`` carries the GPU's own state on the device (for full-size
  runs the oracle cannot follow) and checks, after every step, properties that
  hold at any size: lengths advance by accepted + 1, the emitted offsets are
  the exclusive scan of accepted + 1, every pool page is held by exactly one
  live slot or sits on the free stack, each live slot holds exactly the pages
  its new length needs with its old prefix unchanged, and the compaction keeps
  the survivors in order.
"""
from __future__ import annotations

import numpy as np

from oracle import verify_step as o
import workloads as wl


def _ceil_div(a, b):
    return (a + b - 1) // b


class OracleSwarm:
    def __init__(self, dims, gamma_max, B, pool_pages, ctx, limits, budget, workload=9):
        self.dims, self.gmax, self.B, self.budget, self.wid = dims, gamma_max, B, budget, workload
        self.ctx, self.limits = ctx, limits
        P = dims["page"]
        # a sequence grows by at most its output length before it finishes
        self.max_pages = _ceil_div(ctx[1] + limits[1] + 2 * (gamma_max + 1), P) + 1
        g = wl.rng(workload, wl.S_SEQ, 0)
        self.pool = np.zeros((pool_pages, dims["n_kv"], 2, P, dims["head_dim"]), dtype=np.uint16)
        wl.fill_kv_normal(self.pool, workload)
        self.free = g.permutation(pool_pages).astype(np.int32)
        self.num_free = pool_pages
        self.seq_lens = np.zeros(0, np.int32)
        self.page_table = np.zeros((0, self.max_pages), np.int32)
        self.num_pages = np.zeros(0, np.int32)
        self.gen_counts = np.zeros(0, np.int32)
        self.gen_limits = np.zeros(0, np.int32)
        self.step_no = 0
        self.admitted = 0
        self._admit(B)

    # -- new sequences: fresh length, pages from the free stack top, fresh KV --
    def _admit(self, n):
        P = self.dims["page"]
        g = wl.rng(self.wid, wl.S_SEQ, 1000 + self.step_no)
        lens, rows, lims = [], [], []
        for i in range(n):
            L = int(g.integers(self.ctx[0], self.ctx[1] + 1))
            need = _ceil_div(L + self.gmax + 1, P)
            if need > self.num_free:
                break
            pages = self.free[self.num_free - need:self.num_free][::-1].copy()
            self.num_free -= need
            row = np.full(self.max_pages, -1, np.int32)
            row[:need] = pages
            self.pool[pages] = wl.normal_bf16(wl._key(self.wid, wl.S_KV, 1 + self.admitted), self.pool[pages].shape, 1.0)
            self.admitted += 1
            lens.append(L)
            rows.append(row)
            lims.append(int(wl.loguniform_lengths(g, 1, *self.limits)[0]))
        if lens:
            self.seq_lens = np.concatenate([self.seq_lens, np.array(lens, np.int32)])
            self.page_table = np.concatenate([self.page_table, np.stack(rows)])
            self.num_pages = np.concatenate([self.num_pages, (self.page_table[-len(lens):] >= 0).sum(1).astype(np.int32)])
            self.gen_counts = np.concatenate([self.gen_counts, np.zeros(len(lens), np.int32)])
            self.gen_limits = np.concatenate([self.gen_limits, np.array(lims, np.int32)])

    def batch(self) -> wl.Batch:
        """This step's inputs: the carried state plus fresh drafts, q and uniforms."""
        n = len(self.seq_lens)
        gam = wl.swarm_gamma(n, self.budget, self.gmax)
        draft = np.full(n, gam, np.int32)
        R, G, V = int(n * (gam + 1)), int(n * gam), self.dims["vocab"]
        tokens = wl.rng(self.wid, wl.S_TOKENS, self.step_no).integers(0, V, size=R).astype(np.int32)
        if G:
            ql = wl.rng(self.wid, wl.S_Q, self.step_no).standard_normal((G, V), dtype=np.float32) * np.float32(2.0)
            q = wl.softmax_f32(ql)
        else:
            q = np.zeros((0, V), np.float32)
        u = wl.uniform24(wl.rng(self.wid, wl.S_U, self.step_no), R)
        return wl.Batch(dims=self.dims, gamma_max=self.gmax, seq_lens=self.seq_lens.copy(), draft_lens=draft,
                        tokens=tokens, draft_probs=q, uniforms=u, kv_pool=self.pool.copy(),
                        page_table=self.page_table.copy(), num_pages=self.num_pages.copy(),
                        free_pages=self.free.copy(), num_free=self.num_free, gen_counts=self.gen_counts.copy(),
                        gen_limits=self.gen_limits.copy())

    def advance(self, batch: wl.Batch, ref: dict):
        """Carry the oracle's result: its K/V rows, realignment, compaction, then refill."""
        P = self.dims["page"]
        for (b, pos), (k, v) in ref["forward"]["kv_rows"].items():
            pg = batch.page_table[b, pos // P]
            self.pool[pg, :, 0, pos % P, :] = o.f64_to_bf16_bits(k)
            self.pool[pg, :, 1, pos % P, :] = o.f64_to_bf16_bits(v)
        ra = ref["realign"]
        assert ra["status"] == 0
        src = ra["next_src"]
        self.seq_lens = ra["next_seq_lens"].astype(np.int32)
        self.page_table = ra["next_page_table"].astype(np.int32)
        self.num_pages = ra["next_num_pages"].astype(np.int32)
        self.gen_counts = ra["next_gen_counts"].astype(np.int32)
        self.gen_limits = self.gen_limits[src]
        self.free = ra["free_pages"].astype(np.int32)
        self.num_free = int(ra["num_free"])
        self.step_no += 1
        finished = self.B - len(src)
        self._admit(self.B - len(self.seq_lens))
        return finished


# ---------------------------------------------------------------------------
# the device-carried swarm (full size, invariants only)
# ---------------------------------------------------------------------------

class DeviceSwarm:
    def __init__(self, eng, dims, gamma_max, B, pool_pages, ctx, limits, budget, workload=5):
        import torch
        from workloads import device as wd
        self.eng, self.dims, self.gmax, self.B, self.budget, self.wid = eng, dims, gamma_max, B, budget, workload
        self.ctx, self.limits = ctx, limits
        P = dims["page"]
        # a sequence grows by at most its output length before it finishes
        self.max_pages = _ceil_div(ctx[1] + limits[1] + 2 * (gamma_max + 1), P) + 1
        self.pool = torch.empty((pool_pages, dims["n_kv"], 2, P, dims["head_dim"]), dtype=torch.bfloat16,
                                device="cuda")
        wd.normal_bf16_device_(self.pool, wl._key(workload, wl.S_KV, 0))
        g = wl.rng(workload, wl.S_SEQ, 0)
        self.free = g.permutation(pool_pages).astype(np.int32)
        self.num_free = pool_pages
        self.pool_pages = pool_pages
        self.seq_lens = np.zeros(0, np.int32)
        self.page_table = np.zeros((0, self.max_pages), np.int32)
        self.gen_counts = np.zeros(0, np.int32)
        self.gen_limits = np.zeros(0, np.int32)
        self.step_no = 0
        self.admitted = 0
        self.finished_total = 0
        self.tokens_total = 0
        self._admit(B)

    def _admit(self, n):
        import torch
        from workloads import device as wd
        P = self.dims["page"]
        g = wl.rng(self.wid, wl.S_SEQ, 1000 + self.step_no)
        for _ in range(n):
            L = int(g.integers(self.ctx[0], self.ctx[1] + 1))
            need = _ceil_div(L + self.gmax + 1, P)
            if need > self.num_free:
                break
            pages = self.free[self.num_free - need:self.num_free][::-1].copy()
            self.num_free -= need
            row = np.full(self.max_pages, -1, np.int32)
            row[:need] = pages
            idx = torch.from_numpy(pages.astype(np.int64)).cuda()
            fresh = torch.empty((need,) + tuple(self.pool.shape[1:]), dtype=torch.bfloat16, device="cuda")
            wd.normal_bf16_device_(fresh, wl._key(self.wid, wl.S_KV, 1 + self.admitted))
            self.pool.index_copy_(0, idx, fresh)
            self.admitted += 1
            self.seq_lens = np.append(self.seq_lens, np.int32(L))
            self.page_table = np.concatenate([self.page_table, row[None]])
            self.gen_counts = np.append(self.gen_counts, np.int32(0))
            self.gen_limits = np.append(self.gen_limits, np.int32(wl.loguniform_lengths(g, 1, *self.limits)[0]))

    def inputs(self):
        """Device inputs of this step (drafts, q and uniforms drawn fresh)."""
        import torch
        from workloads import device as wd
        n = len(self.seq_lens)
        gam = wl.swarm_gamma(n, self.budget, self.gmax)
        R, G, V = n * (gam + 1), n * gam, self.dims["vocab"]
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        num_pages = (self.page_table >= 0).sum(1).astype(np.int32)
        bd = dict(B=n, R=R, G=G, seq_lens=t(self.seq_lens), draft_lens=t(np.full(n, gam, np.int32)),
                  tokens=t(wl.rng(self.wid, wl.S_TOKENS, self.step_no).integers(0, V, size=R).astype(np.int32)),
                  draft_probs=wd.draft_probs_device(G, V, wl._key(self.wid, wl.S_Q, self.step_no)),
                  uniforms=t(wl.uniform24(wl.rng(self.wid, wl.S_U, self.step_no), R)),
                  kv_pool=self.pool, num_pool_pages=self.pool_pages, page_table=t(self.page_table),
                  num_pages=t(num_pages), free_pages=t(self.free), num_free_in=t(np.array([self.num_free], np.int32)),
                  gen_counts=t(self.gen_counts), gen_limits=t(self.gen_limits))
        bd["num_free_out"] = bd["num_free_in"]
        return bd

    def step(self, bd=None, res=None):
        """One verify step on the carried state, the invariant checks, then compaction + refill."""
        import torch
        from workloads import device as wd
        if bd is None:
            bd = self.inputs()
        n, R = bd["B"], bd["R"]
        if res is None:
            res = wd.alloc_result(n, R, self.dims["vocab"], self.gmax, self.max_pages)
        self.eng.verify_step(bd, res)
        assert self.eng.read_status(res["status"]) == 0
        torch.cuda.synchronize()
        c = lambda k: res[k].cpu().numpy()  # noqa: E731
        acc, new_len, fin = c("accepted"), c("new_seq_lens"), c("finished").astype(bool)
        gam = int(bd["draft_lens"][0].item()) if n else 0
        old_pt = self.page_table
        # lengths, counts, emitted offsets
        assert np.all((acc >= 0) & (acc <= gam))
        assert np.array_equal(new_len, self.seq_lens + acc + 1)
        eoff = c("emitted_offsets")
        assert eoff[0] == 0 and np.array_equal(np.diff(eoff), acc + 1)
        new_gen = self.gen_counts + acc + 1
        assert np.array_equal(fin, new_gen >= self.gen_limits)
        # compaction: survivors in order, their state gathered
        nl = int(c("num_live")[0])
        src = c("next_src")[:nl]
        assert np.array_equal(src, np.nonzero(~fin)[0])
        nsl = c("next_seq_lens")[:nl]
        npt = c("next_page_table")[:nl]
        nnp = c("next_num_pages")[:nl]
        assert np.array_equal(nsl, new_len[src])
        assert np.array_equal(c("next_gen_counts")[:nl], new_gen[src])
        P = self.dims["page"]
        need = _ceil_div(nsl + self.gmax + 1, P)
        assert np.array_equal(nnp, need)
        for j, s in enumerate(src):
            keep = min(int(need[j]), int((old_pt[s] >= 0).sum()))
            assert np.array_equal(npt[j, :keep], old_pt[s, :keep])
            assert np.all(npt[j, need[j]:] == -1) and np.all(npt[j, :need[j]] >= 0)
        # every pool page held by one live slot or on the free stack, once
        nf = int(bd["num_free_out"].cpu().numpy()[0])
        free = bd["free_pages"].cpu().numpy()[:nf]
        held = np.concatenate([npt[j, :need[j]] for j in range(nl)] + [free])
        assert np.array_equal(np.sort(held), np.arange(self.pool_pages))
        # carry the GPU's state, refill the freed slots
        self.tokens_total += int(eoff[-1])
        self.finished_total += int(fin.sum())
        self.seq_lens = nsl.astype(np.int32)
        self.page_table = np.full((nl, self.max_pages), -1, np.int32)
        self.page_table[:, :npt.shape[1]] = npt
        self.gen_counts = new_gen[src].astype(np.int32)
        self.gen_limits = self.gen_limits[src]
        self.free = bd["free_pages"].cpu().numpy().astype(np.int32)
        self.num_free = nf
        self.step_no += 1
        self._admit(self.B - nl)
        return res, acc


def host_sub_batch(bd: dict, slots, dims, gamma_max) -> tuple:
    """Host copy of the inputs of some slots of a device batch (read before the step):
    lengths, drafts, tokens, q rows, uniforms and their KV pages, renumbered into a
    compact pool.  Returns the sub-batch, the global row index of each of its rows,
    and the pool pages it holds (in compact order)."""
    import torch
    c = lambda k: bd[k].cpu().numpy()  # noqa: E731
    seq_lens, draft = c("seq_lens"), c("draft_lens")
    roff = wl.row_offsets(draft)
    goff = np.concatenate([[0], np.cumsum(draft)])
    pt = c("page_table")
    rows, grows, pages = [], [], []
    for s in slots:
        rows.extend(range(int(roff[s]), int(roff[s + 1])))
        grows.extend(range(int(goff[s]), int(goff[s + 1])))
        pages.append(pt[s][pt[s] >= 0])
    allp = np.concatenate(pages).astype(np.int64)
    pool = read_pages(bd["kv_pool"], allp)
    new_pt = np.full((len(slots), pt.shape[1]), -1, np.int32)
    o_ = 0
    for i, p in enumerate(pages):
        new_pt[i, :len(p)] = np.arange(o_, o_ + len(p))
        o_ += len(p)
    if grows:
        q = bd["draft_probs"][torch.from_numpy(np.array(grows, np.int64)).cuda()].cpu().numpy()
    else:
        q = np.zeros((0, dims["vocab"]), np.float32)
    sub = wl.Batch(dims=dims, gamma_max=gamma_max, seq_lens=seq_lens[slots], draft_lens=draft[slots],
                   tokens=c("tokens")[rows], draft_probs=q, uniforms=c("uniforms")[rows], kv_pool=pool,
                   page_table=new_pt, num_pages=(new_pt >= 0).sum(1).astype(np.int32),
                   free_pages=np.zeros(0, np.int32), num_free=0)
    return sub, np.array(rows, np.int64), allp


def read_pages(pool, pages) -> np.ndarray:
    """bf16 bits of the given pool pages, in that order."""
    import torch
    idx = torch.from_numpy(np.asarray(pages, dtype=np.int64)).cuda()
    return pool[idx].view(torch.int16).cpu().numpy().view(np.uint16)
