"""Continuous-batching verify loop: the scheduler, admission and the verify step.

One ``SwarmRunner.step()`` is one iteration of the loop the pages describe for
an agent swarm ("Why Static Batching Wastes an RX 9070 XT Agent Swarm and
Continuous Batching Wins It Back", "Continuous batching refills the slot
instead of freezing it"; "Speculative Decoding and Batching Compete for the
Same Compute Slack on RDNA4", "What the budget says to build"):

  1. the host scheduler (C++) admits queued sequences into free slots and picks
     the draft length from the live batch size;
  2. ``sdv_admit`` appends the newcomers to the device slot table;
  3. the caller's drafter fills tokens, draft probabilities and uniforms;
  4. ``sdv_verify_step`` verifies, samples and realigns every slot on the GPU,
     writing the compacted next-slot view into the other of two slot tables;
  5. the accepted counts come back to the host and the scheduler retires the
     finished sequences.

This module only marshals arguments and moves the few per-step integers; the
state changes happen in the library.
"""
from __future__ import annotations

from . import VerifyEngine
from .sched import CONTINUOUS, Scheduler


class SwarmRunner:
    def __init__(self, engine: VerifyEngine, kv_pool, pool_pages: int, max_slots: int, budget_rows: int,
                 max_pages_per_seq: int, free_order=None, policy: int = CONTINUOUS):
        import torch
        cfg = engine.cfg_dict
        self.eng = engine
        self.V = int(cfg["vocab"])
        self.gamma_max = int(cfg["gamma_max"])
        self.page = int(cfg.get("page_size", 16))
        self.kv_pool = kv_pool
        self.pool_pages = int(pool_pages)
        self.max_slots = int(max_slots)
        self.max_pages = int(max_pages_per_seq)
        self.sched = Scheduler(max_slots, self.gamma_max, budget_rows, pool_pages, max_pages_per_seq,
                               page_size=self.page, policy=policy)
        dev = "cuda"
        i32 = dict(dtype=torch.int32, device=dev)

        def table():
            return dict(seq_lens=torch.zeros(max_slots, **i32), num_pages=torch.zeros(max_slots, **i32),
                        gen_counts=torch.zeros(max_slots, **i32), gen_limits=torch.zeros(max_slots, **i32),
                        page_table=torch.full((max_slots, max_pages_per_seq), -1, **i32))

        self.tables = [table(), table()]
        order = torch.arange(pool_pages, **i32) if free_order is None else free_order.to(dev, torch.int32)
        self.free_pages = order.clone()
        self.num_free = torch.tensor([pool_pages], **i32)
        self.status = torch.zeros(1, **i32)
        R = max_slots * (self.gamma_max + 1)
        self.res = dict(accepted=torch.zeros(max_slots, **i32), final_tokens=torch.zeros(max_slots, **i32),
                        emitted_tokens=torch.zeros(R, **i32), emitted_offsets=torch.zeros(max_slots + 1, **i32),
                        new_seq_lens=torch.zeros(max_slots, **i32), finished=torch.zeros(max_slots, **i32),
                        new_gen_counts=torch.zeros(max_slots, **i32), next_src=torch.zeros(max_slots, **i32),
                        num_live=torch.zeros(1, **i32), status=self.status)
        self.draft_lens = torch.zeros(max_slots, **i32)
        # pinned host copies of the per-step integers that come back
        self._acc_host = torch.zeros(max_slots, dtype=torch.int32, pin_memory=True)
        self._status_host = torch.zeros(1, dtype=torch.int32, pin_memory=True)
        self.k = 0
        self.have_prev = False
        self.last = None

    def submit(self, seq_id: int, ctx_len: int, out_len: int):
        self.sched.submit(seq_id, ctx_len, out_len)

    def plan(self) -> dict:
        """Scheduler decision + device admission for the next step; returns the plan
        and the device batch dict (without the drafter's tokens / q / uniforms)."""
        import torch
        st = self.sched.plan()
        t_in, t_prev = self.tables[self.k % 2], self.tables[(self.k + 1) % 2]
        survivors = st["live"] - st["admitted"]
        n = st["admitted"]
        ctx = torch.tensor(st["admit_ctx"], dtype=torch.int32).cuda(non_blocking=True) if n else None
        out = torch.tensor(st["admit_out"], dtype=torch.int32).cuda(non_blocking=True) if n else None
        prev = dict(num_live=self.res["num_live"], next_src=self.res["next_src"],
                    gen_limits_prev=t_prev["gen_limits"]) if self.have_prev else {}
        if n or prev:
            self.eng.admit(t_in, survivors, ctx, out, self.free_pages, self.num_free, self.status, **prev)
        B = st["live"]
        if B:
            self.draft_lens[:B].fill_(st["gamma"])
        batch = dict(B=B, R=st["rows"], G=st["drafts"], seq_lens=t_in["seq_lens"], draft_lens=self.draft_lens,
                     kv_pool=self.kv_pool, num_pool_pages=self.pool_pages, page_table=t_in["page_table"],
                     num_pages=t_in["num_pages"], free_pages=self.free_pages, num_free_in=self.num_free,
                     num_free_out=self.num_free, gen_counts=t_in["gen_counts"], gen_limits=t_in["gen_limits"])
        return st, batch

    def verify(self, st: dict, batch: dict, stream=None):
        """Enqueue the verify step of a planned batch (drafts filled in by the caller)."""
        t_out = self.tables[(self.k + 1) % 2]
        r = dict(self.res)
        r.update(next_seq_lens=t_out["seq_lens"], next_num_pages=t_out["num_pages"],
                 next_page_table=t_out["page_table"], next_gen_counts=t_out["gen_counts"])
        self.eng.verify_step(batch, r, stream)

    def complete(self, st: dict) -> list:
        """Bring the accepted counts back and let the scheduler retire the finished."""
        import torch
        from . import SdvError
        B = st["live"]
        self._acc_host[:B].copy_(self.res["accepted"][:B], non_blocking=True)
        self._status_host.copy_(self.status, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if int(self._status_host[0]) != 0:
            raise SdvError(int(self._status_host[0]), "device status after the verify step")
        fin = self.sched.complete(self._acc_host[:B].tolist())
        self.k += 1
        self.have_prev = True
        self.last = st
        return fin

    def step(self, drafter, stream=None):
        """plan -> drafter(st, batch) fills tokens / draft_probs / uniforms -> verify -> complete."""
        st, batch = self.plan()
        if st["live"] == 0:
            return st, []
        drafter(st, batch)
        self.verify(st, batch, stream)
        return st, self.complete(st)

    def table(self):
        """The device slot table the next step reads (after the last step's compaction)."""
        return self.tables[self.k % 2]
