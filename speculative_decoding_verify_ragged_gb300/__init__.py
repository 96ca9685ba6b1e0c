"""Ragged batched speculative-verify step on GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/sdv.h``: it converts torch
tensors and dicts into the ABI's structs and calls the CUDA library.  Every
step of the verify path (weight-streaming GEMMs with fused epilogues, paged
ragged attention, LM head and softmax statistics, rejection-sampling
acceptance, realignment) runs in the library's kernels; if the library is
missing the calls raise, there is no CPU path.

Typical use::

    eng = VerifyEngine(cfg, weights, max_rows=64, max_slots=8)
    eng.verify_step(batch, result)          # enqueued on the current stream
    status = eng.read_status(result["status"])
"""
from __future__ import annotations

import ctypes

from ._abi import (PHASES, RESULT_FIELDS, STATUS, SDV_OK, SDV_WEIGHTS_BF16, SDV_WEIGHTS_INT4_G32, SdvAdmission,
                   SdvBatch, SdvConfig, SdvResult, SdvWeights, load_library)

__all__ = ["VerifyEngine", "SdvError", "PHASES", "STATUS", "load_library", "kernel_launches", "SDV_WEIGHTS_BF16",
           "SDV_WEIGHTS_INT4_G32"]


class SdvError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def kernel_launches() -> int:
    return int(load_library().sdv_kernel_launches())


CONFIG_KEYS = ("hidden", "n_q", "n_kv", "head_dim", "ffn", "vocab", "page_size", "gamma_max", "weight_format")
WEIGHT_KEYS = ("emb", "w_qkv", "w_o", "w_gate", "w_up", "w_down", "w_lm", "s_qkv", "s_o", "s_gate", "s_up",
               "s_down", "g_attn", "g_ffn", "g_final")


class VerifyEngine:
    """A verify-step context over device-resident weights.

    cfg: dict with the sdv_config fields (rms_eps / rope_theta default to
    1e-6 / 1e6).  weights: dict of CUDA tensors named as sdv_weights.  The
    workspace is allocated here through torch (the library never allocates).
    """

    def __init__(self, cfg: dict, weights: dict, max_rows: int, max_slots: int, lib_path: str | None = None):
        import torch
        self.lib = load_library(lib_path) if lib_path else load_library()
        self.cfg_dict = dict(cfg)
        self.cfg = SdvConfig(*[int(cfg.get(k, 0)) for k in CONFIG_KEYS],
                             float(cfg.get("rms_eps", 1e-6)), float(cfg.get("rope_theta", 1e6)))
        self._weights = {k: weights.get(k) for k in WEIGHT_KEYS}   # keep tensors alive
        self.wstruct = SdvWeights(*[_ptr(self._weights[k]) for k in WEIGHT_KEYS])
        self.max_rows = int(max_rows)
        self.max_slots = int(max_slots)
        nbytes = self.lib.sdv_workspace_size(ctypes.byref(self.cfg), self.max_rows, self.max_slots)
        if nbytes == 0:
            raise SdvError(1, "sdv_workspace_size rejected the configuration")
        self.workspace = torch.empty(int(nbytes), dtype=torch.uint8, device="cuda")
        self.workspace_bytes = int(nbytes)
        h = ctypes.c_void_p()
        rc = self.lib.sdv_create(ctypes.byref(self.cfg), ctypes.byref(self.wstruct), _ptr(self.workspace),
                                 ctypes.c_size_t(nbytes), self.max_rows, self.max_slots, ctypes.byref(h))
        if rc != SDV_OK:
            raise SdvError(rc, "sdv_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.sdv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- marshalling -------------------------------------------------------

    @staticmethod
    def batch_struct(b: dict) -> SdvBatch:
        pt = b["page_table"]
        return SdvBatch(int(b["B"]), int(b["R"]), int(b["G"]),
                        _ptr(b["seq_lens"]), _ptr(b["draft_lens"]), _ptr(b.get("tokens")),
                        _ptr(b.get("draft_probs")), _ptr(b.get("uniforms")),
                        _ptr(b.get("kv_pool")), int(b.get("num_pool_pages", 0)),
                        _ptr(pt), int(pt.shape[1]),
                        _ptr(b["num_pages"]), _ptr(b.get("free_pages")),
                        _ptr(b.get("num_free_in")), _ptr(b.get("num_free_out")),
                        _ptr(b.get("gen_counts")), _ptr(b.get("gen_limits")), _ptr(b.get("tree_parents")))

    @staticmethod
    def result_struct(r: dict) -> SdvResult:
        return SdvResult(*[_ptr(r.get(k)) for k in RESULT_FIELDS])

    def _check(self, rc, what):
        if rc != SDV_OK:
            extra = ""
            if rc == 4:
                extra = f" (cuda error {self.lib.sdv_last_cuda_error()})"
            raise SdvError(rc, what + extra)

    # -- entry points ------------------------------------------------------

    def verify_step(self, batch: dict, result: dict, stream=None):
        bs, rs = self.batch_struct(batch), self.result_struct(result)
        self._check(self.lib.sdv_verify_step(self.handle, ctypes.byref(bs), ctypes.byref(rs), _stream(stream)),
                    "sdv_verify_step")

    def accept(self, probs, batch: dict, result: dict, stream=None):
        bs, rs = self.batch_struct(batch), self.result_struct(result)
        self._check(self.lib.sdv_accept(self.handle, _ptr(probs), ctypes.byref(bs), ctypes.byref(rs),
                                        _stream(stream)), "sdv_accept")

    def realign(self, batch: dict, result: dict, stream=None):
        bs, rs = self.batch_struct(batch), self.result_struct(result)
        self._check(self.lib.sdv_realign(self.handle, ctypes.byref(bs), ctypes.byref(rs), _stream(stream)),
                    "sdv_realign")

    def linear(self, which: int, x, y, stream=None):
        """y = x W^T (fp32); x bf16 or fp32 [rows, K]."""
        import torch
        fmt = 1 if x.dtype == torch.float32 else 0
        self._check(self.lib.sdv_linear(self.handle, int(which), _ptr(x), fmt, _ptr(y), int(x.shape[0]),
                                        _stream(stream)), "sdv_linear")

    def attention(self, q, batch: dict, out, status, stream=None):
        bs = self.batch_struct(batch)
        self._check(self.lib.sdv_attention(self.handle, _ptr(q), ctypes.byref(bs), _ptr(out), _ptr(status),
                                           _stream(stream)), "sdv_attention")

    def admit(self, table: dict, live: int, ctx_lens, out_lens, free_pages, num_free, status,
              num_live=None, next_src=None, gen_limits_prev=None, stream=None):
        """Append newcomers to a device slot table (sdv_admit).

        table: dict of device int32 tensors seq_lens, num_pages, gen_counts,
        gen_limits [slots] and page_table [slots, max_pages]; ctx_lens /
        out_lens: device int32 [n]."""
        pt = table["page_table"]
        n = 0 if ctx_lens is None else int(ctx_lens.numel())
        a = SdvAdmission(int(live), n, int(pt.shape[0]), _ptr(num_live), _ptr(next_src), _ptr(gen_limits_prev),
                         _ptr(ctx_lens), _ptr(out_lens), _ptr(table["seq_lens"]), _ptr(table["num_pages"]),
                         _ptr(table["gen_counts"]), _ptr(table["gen_limits"]), _ptr(pt), int(pt.shape[1]),
                         _ptr(free_pages), _ptr(num_free))
        self._check(self.lib.sdv_admit(self.handle, ctypes.byref(a), _ptr(status), _stream(stream)), "sdv_admit")

    def set_gemm_path(self, path: int):
        """0 auto (by row count), 1 bf16 mma.sync, 2 tcgen05 with TMEM accumulators."""
        self._check(self.lib.sdv_set_gemm_path(self.handle, int(path)), "sdv_set_gemm_path")

    def set_sampling(self, mode: int):
        """0 stochastic (rejection sampling, default), 1 greedy (argmax tests and final token)."""
        self._check(self.lib.sdv_set_sampling(self.handle, int(mode)), "sdv_set_sampling")

    def set_trace(self, table):
        """Point the step timeline at a device int64 tensor [32, 3] (None stops
        it); only the timeline build libsdv_trace.so accepts it."""
        self._check(self.lib.sdv_trace_enable(_ptr(table)), "sdv_trace_enable")

    def set_attention_path(self, path: int):
        """0 auto, 1 mma.sync (<= 48 query vectors per sequence and kv head), 2 tcgen05
        (head_dim 128, <= 64 query vectors: <= 48 in one work item, 32 per item past 48)."""
        self._check(self.lib.sdv_set_attention_path(self.handle, int(path)), "sdv_set_attention_path")

    def set_stall_test(self, stall_ns: int):
        """Test hook: > 0 makes the next calls' first kernel give up a wait that
        nothing ends after stall_ns and report SDV_ERR_TIMEOUT; 0 turns it off."""
        self._check(self.lib.sdv_set_stall_test(self.handle, int(stall_ns)), "sdv_set_stall_test")

    def set_phase_events(self, events):
        """Record torch.cuda.Event objects at the step's phase boundaries (None = off).

        ``events`` holds len(PHASES) + 1 events created with enable_timing=True, or None
        for boundaries not to record (each recorded event blocks the overlap of the two
        kernels it separates).
        """
        if events is None:
            self._check(self.lib.sdv_set_phase_events(self.handle, None, 0), "sdv_set_phase_events")
            self._events = None
            return
        for e in events:
            if e is not None and not e.cuda_event:
                e.record()          # creates the underlying CUDA event
        arr = (ctypes.c_void_p * len(events))(*[(e.cuda_event if e is not None else None) for e in events])
        self._events = list(events)
        self._check(self.lib.sdv_set_phase_events(self.handle, arr, len(events)), "sdv_set_phase_events")

    def read_status(self, status, stream=None) -> int:
        """The step's status word, read through this engine's library (the
        timeline build may be the only one present)."""
        out = ctypes.c_int(-1)
        rc = self.lib.sdv_read_status(_ptr(status), ctypes.byref(out), _stream(stream))
        if rc != SDV_OK:
            raise SdvError(rc, "sdv_read_status")
        return int(out.value)
