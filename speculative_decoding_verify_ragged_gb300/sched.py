"""Python binding of the host-side continuous-batching scheduler (``include/sdv_sched.h``).

Argument marshalling only: the policy (draft length from the live batch and a
row budget, admission from an arrival-order queue, retirement and stable
compaction) runs in the library's C++ code.
"""
from __future__ import annotations

import ctypes

from ._abi import (SDV_OK, SDV_SCHED_CONTINUOUS, SDV_SCHED_STATIC, SDV_SCHED_STATIC_SHRINK, SdvSchedConfig,
                   SdvSchedStats, SdvSchedStep, load_library)

__all__ = ["Scheduler", "draft_length", "CONTINUOUS", "STATIC", "STATIC_SHRINK"]

CONTINUOUS, STATIC, STATIC_SHRINK = SDV_SCHED_CONTINUOUS, SDV_SCHED_STATIC, SDV_SCHED_STATIC_SHRINK


def draft_length(budget_rows: int, live: int, gamma_max: int) -> int:
    """The budget rule: clamp((budget - live) // live, 0, gamma_max)."""
    return int(load_library().sdv_sched_gamma(int(budget_rows), int(live), int(gamma_max)))


class Scheduler:
    """Slot membership and draft length of every step, mirrored on the host.

    ``plan()`` admits queued sequences and picks gamma; ``complete(accepted)``
    advances the live sequences by accepted + 1 and retires the finished ones,
    exactly as the device realignment does, so the device slot table and this
    mirror stay equal step after step.
    """

    def __init__(self, max_slots: int, gamma_max: int, budget_rows: int, pool_pages: int,
                 max_pages_per_seq: int, page_size: int = 16, policy: int = CONTINUOUS):
        from . import SdvError
        self.lib = load_library()
        self.cfg = SdvSchedConfig(int(max_slots), int(gamma_max), int(budget_rows), int(page_size),
                                  int(pool_pages), int(max_pages_per_seq), int(policy))
        h = ctypes.c_void_p()
        rc = self.lib.sdv_sched_create(ctypes.byref(self.cfg), ctypes.byref(h))
        if rc != SDV_OK:
            raise SdvError(rc, "sdv_sched_create")
        self.handle = h
        n = int(max_slots)
        self._ctx = (ctypes.c_int * n)()
        self._out = (ctypes.c_int * n)()
        self._ids = (ctypes.c_longlong * n)()
        self._fin = (ctypes.c_longlong * n)()
        self._acc = (ctypes.c_int * n)()
        self.step = None

    def close(self):
        if getattr(self, "handle", None):
            self.lib.sdv_sched_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, rc, what):
        from . import SdvError
        if rc != SDV_OK:
            raise SdvError(rc, what)

    def submit(self, seq_id: int, ctx_len: int, out_len: int):
        self._check(self.lib.sdv_sched_submit(self.handle, int(seq_id), int(ctx_len), int(out_len)),
                    "sdv_sched_submit")

    def plan(self) -> dict:
        """Next step: live, width, gamma, rows, drafts, admitted, plus the
        admitted sequences' (ctx_len, out_len) lists and the live slots' ids."""
        st = SdvSchedStep()
        self._check(self.lib.sdv_sched_plan(self.handle, ctypes.byref(st), self._ctx, self._out, self._ids),
                    "sdv_sched_plan")
        d = {k: int(getattr(st, k)) for k, _ in SdvSchedStep._fields_}
        d["admit_ctx"] = [int(self._ctx[i]) for i in range(st.admitted)]
        d["admit_out"] = [int(self._out[i]) for i in range(st.admitted)]
        d["ids"] = [int(self._ids[i]) for i in range(st.live)]
        self.step = d
        return d

    def complete(self, accepted) -> list:
        """Account the planned step from its accepted counts; returns the retired ids."""
        acc = [int(a) for a in accepted]
        for i, a in enumerate(acc):
            self._acc[i] = a
        n = ctypes.c_int(0)
        self._check(self.lib.sdv_sched_complete(self.handle, self._acc, self._fin, ctypes.byref(n)),
                    "sdv_sched_complete")
        return [int(self._fin[i]) for i in range(n.value)]

    def stats(self) -> dict:
        st = SdvSchedStats()
        self._check(self.lib.sdv_sched_get_stats(self.handle, ctypes.byref(st)), "sdv_sched_get_stats")
        return {k: int(getattr(st, k)) for k, _ in SdvSchedStats._fields_}

    def slots(self) -> dict:
        """Host mirror of the live slots: seq_lens, gen_counts, out_lens, num_pages (slot order)."""
        n = int(self.cfg.max_slots)
        arrs = [(ctypes.c_int * n)() for _ in range(4)]
        self._check(self.lib.sdv_sched_slots(self.handle, *arrs), "sdv_sched_slots")
        live = self.stats()["live"]
        keys = ("seq_lens", "gen_counts", "out_lens", "num_pages")
        return {k: [int(a[i]) for i in range(live)] for k, a in zip(keys, arrs)}
