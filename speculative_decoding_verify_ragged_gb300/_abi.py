"""ctypes mirror of include/sdv.h and the loader of the in-tree ``libsdv.so``.

Argument marshalling only: every step of the verify path runs in the CUDA
library.  A missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsdv.so")

c_int = ctypes.c_int
c_float = ctypes.c_float
c_void_p = ctypes.c_void_p
c_size_t = ctypes.c_size_t

STATUS = {
    0: "SDV_OK",
    1: "SDV_ERR_INVALID_ARG",
    2: "SDV_ERR_CAPACITY",
    3: "SDV_ERR_PAGE_RANGE",
    4: "SDV_ERR_CUDA",
    5: "SDV_ERR_TIMEOUT",
    6: "SDV_ERR_BAD_INPUT",
    7: "SDV_ERR_UNSUPPORTED",
    8: "SDV_ERR_INTERNAL",
}
SDV_OK, SDV_ERR_INVALID_ARG, SDV_ERR_CAPACITY, SDV_ERR_PAGE_RANGE, SDV_ERR_CUDA, SDV_ERR_TIMEOUT, \
    SDV_ERR_BAD_INPUT, SDV_ERR_UNSUPPORTED, SDV_ERR_INTERNAL = range(9)
SDV_WEIGHTS_BF16, SDV_WEIGHTS_INT4_G32 = 0, 1
SDV_GEMM_AUTO, SDV_GEMM_MMA_SYNC, SDV_GEMM_TCGEN05 = 0, 1, 2
SDV_SAMPLING_STOCHASTIC, SDV_SAMPLING_GREEDY = 0, 1
PHASES = ("prologue", "qkv", "attention", "o_proj", "ffn", "lm_head", "accept", "realign")


class SdvConfig(ctypes.Structure):
    _fields_ = [(n, c_int) for n in ("hidden", "n_q", "n_kv", "head_dim", "ffn", "vocab", "page_size",
                                     "gamma_max", "weight_format")] + [("rms_eps", c_float), ("rope_theta", c_float)]


class SdvWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("emb", "w_qkv", "w_o", "w_gate", "w_up", "w_down", "w_lm",
                                        "s_qkv", "s_o", "s_gate", "s_up", "s_down",
                                        "g_attn", "g_ffn", "g_final")]


class SdvBatch(ctypes.Structure):
    _fields_ = [("B", c_int), ("R", c_int), ("G", c_int),
                ("seq_lens", c_void_p), ("draft_lens", c_void_p), ("tokens", c_void_p),
                ("draft_probs", c_void_p), ("uniforms", c_void_p),
                ("kv_pool", c_void_p), ("num_pool_pages", c_int),
                ("page_table", c_void_p), ("max_pages_per_seq", c_int),
                ("num_pages", c_void_p), ("free_pages", c_void_p),
                ("num_free_in", c_void_p), ("num_free_out", c_void_p),
                ("gen_counts", c_void_p), ("gen_limits", c_void_p), ("tree_parents", c_void_p)]


RESULT_FIELDS = ("accepted", "final_tokens", "emitted_tokens", "emitted_offsets", "new_seq_lens",
                 "finished", "new_gen_counts",
                 "next_src", "num_live", "next_seq_lens", "next_num_pages", "next_page_table", "next_gen_counts",
                 "accept_tested", "accept_accepted", "logits", "probs", "status")


class SdvResult(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in RESULT_FIELDS]


class SdvAdmission(ctypes.Structure):
    _fields_ = [("live", c_int), ("n", c_int), ("slots", c_int),
                ("num_live", c_void_p), ("next_src", c_void_p), ("gen_limits_prev", c_void_p),
                ("ctx_lens", c_void_p), ("out_lens", c_void_p),
                ("seq_lens", c_void_p), ("num_pages", c_void_p), ("gen_counts", c_void_p), ("gen_limits", c_void_p),
                ("page_table", c_void_p), ("max_pages_per_seq", c_int),
                ("free_pages", c_void_p), ("num_free", c_void_p)]


SDV_SCHED_CONTINUOUS, SDV_SCHED_STATIC, SDV_SCHED_STATIC_SHRINK = 0, 1, 2


class SdvSchedConfig(ctypes.Structure):
    _fields_ = [(n, c_int) for n in ("max_slots", "gamma_max", "budget_rows", "page_size", "pool_pages",
                                     "max_pages_per_seq", "policy")]


class SdvSchedStep(ctypes.Structure):
    _fields_ = [(n, c_int) for n in ("live", "width", "gamma", "rows", "drafts", "admitted")]


class SdvSchedStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_longlong) for n in ("steps", "emitted", "slot_steps_paid", "slot_steps_live",
                                                 "finished", "admitted")] + [("queued", c_int), ("free_pages", c_int), ("live", c_int)]


TRACE_LIB_PATH = os.path.join(HERE, "libsdv_trace.so")
_libs: dict = {}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsdv.so (built by ``build.py``), or another build of it such as
    the timeline build libsdv_trace.so; raise if it is not there."""
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run python -m speculative_decoding_verify_ragged_gb300.build)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.sdv_workspace_size.restype = c_size_t
    lib.sdv_workspace_size.argtypes = [P(SdvConfig), c_int, c_int]
    lib.sdv_create.restype = c_int
    lib.sdv_create.argtypes = [P(SdvConfig), P(SdvWeights), c_void_p, c_size_t, c_int, c_int, P(c_void_p)]
    lib.sdv_destroy.restype = None
    lib.sdv_destroy.argtypes = [c_void_p]
    lib.sdv_verify_step.restype = c_int
    lib.sdv_verify_step.argtypes = [c_void_p, P(SdvBatch), P(SdvResult), c_void_p]
    lib.sdv_accept.restype = c_int
    lib.sdv_accept.argtypes = [c_void_p, c_void_p, P(SdvBatch), P(SdvResult), c_void_p]
    lib.sdv_accept_static.restype = c_int
    lib.sdv_accept_static.argtypes = [P(SdvConfig), c_void_p, P(SdvBatch), P(SdvResult), c_void_p]
    lib.sdv_realign.restype = c_int
    lib.sdv_realign.argtypes = [c_void_p, P(SdvBatch), P(SdvResult), c_void_p]
    lib.sdv_linear.restype = c_int
    lib.sdv_linear.argtypes = [c_void_p, c_int, c_void_p, c_int, c_void_p, c_int, c_void_p]
    lib.sdv_attention.restype = c_int
    lib.sdv_attention.argtypes = [c_void_p, c_void_p, P(SdvBatch), c_void_p, c_void_p, c_void_p]
    lib.sdv_set_gemm_path.restype = c_int
    lib.sdv_set_gemm_path.argtypes = [c_void_p, c_int]
    lib.sdv_set_sampling.restype = c_int
    lib.sdv_set_sampling.argtypes = [c_void_p, c_int]
    lib.sdv_set_attention_path.restype = c_int
    lib.sdv_set_attention_path.argtypes = [c_void_p, c_int]
    lib.sdv_set_stall_test.restype = c_int
    lib.sdv_set_stall_test.argtypes = [c_void_p, ctypes.c_ulonglong]
    lib.sdv_set_phase_events.restype = c_int
    lib.sdv_set_phase_events.argtypes = [c_void_p, P(c_void_p), c_int]
    lib.sdv_read_status.restype = c_int
    lib.sdv_read_status.argtypes = [c_void_p, P(c_int), c_void_p]
    lib.sdv_last_cuda_error.restype = c_int
    lib.sdv_last_cuda_error.argtypes = []
    lib.sdv_kernel_launches.restype = ctypes.c_ulonglong
    lib.sdv_kernel_launches.argtypes = []
    lib.sdv_trace_enable.restype = c_int
    lib.sdv_trace_enable.argtypes = [c_void_p]
    lib.sdv_admit.restype = c_int
    lib.sdv_admit.argtypes = [c_void_p, P(SdvAdmission), c_void_p, c_void_p]
    c_ll = ctypes.c_longlong
    lib.sdv_ngram_draft.restype = c_int
    lib.sdv_ngram_draft.argtypes = [P(c_int), c_int, c_int, c_int, c_int, P(c_int)]
    lib.sdv_ngram_draft_batch.restype = c_int
    lib.sdv_ngram_draft_batch.argtypes = [P(c_int), P(c_ll), c_int, c_int, c_int, c_int, P(c_int), P(c_int)]
    lib.sdv_sched_gamma.restype = c_int
    lib.sdv_sched_gamma.argtypes = [c_int, c_int, c_int]
    lib.sdv_sched_create.restype = c_int
    lib.sdv_sched_create.argtypes = [P(SdvSchedConfig), P(c_void_p)]
    lib.sdv_sched_destroy.restype = None
    lib.sdv_sched_destroy.argtypes = [c_void_p]
    lib.sdv_sched_submit.restype = c_int
    lib.sdv_sched_submit.argtypes = [c_void_p, c_ll, c_int, c_int]
    lib.sdv_sched_plan.restype = c_int
    lib.sdv_sched_plan.argtypes = [c_void_p, P(SdvSchedStep), P(c_int), P(c_int), P(c_ll)]
    lib.sdv_sched_complete.restype = c_int
    lib.sdv_sched_complete.argtypes = [c_void_p, P(c_int), P(c_ll), P(c_int)]
    lib.sdv_sched_get_stats.restype = c_int
    lib.sdv_sched_get_stats.argtypes = [c_void_p, P(SdvSchedStats)]
    lib.sdv_sched_slots.restype = c_int
    lib.sdv_sched_slots.argtypes = [c_void_p, P(c_int), P(c_int), P(c_int), P(c_int)]
    _libs[path] = lib
    return lib


def header_symbols(header: str) -> list[str]:
    """Names of the functions declared in a C header (``sdv_*(...)``)."""
    import re
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdv_[a-z_0-9]+)\s*\(", text)))
