"""Python binding of the host n-gram drafter (``include/sdv_draft.h``).

Argument marshalling only; the search runs in the library's C++ code.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._abi import SDV_OK, load_library

__all__ = ["ngram_draft", "ngram_draft_batch"]


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def ngram_draft(history, gamma: int, min_n: int = 1, max_n: int = 4) -> np.ndarray:
    """Drafts for one sequence: the tokens that followed the most recent earlier
    occurrence of its longest matching suffix (max_n down to min_n), up to gamma."""
    h = np.ascontiguousarray(history, dtype=np.int32)
    out = np.zeros(max(gamma, 1), dtype=np.int32)
    k = load_library().sdv_ngram_draft(_ip(h), int(h.size), int(min_n), int(max_n), int(gamma), _ip(out))
    if k < 0:
        raise ValueError("sdv_ngram_draft: bad argument")
    return out[:k].copy()


def ngram_draft_batch(histories, gamma_max: int, min_n: int = 1, max_n: int = 4):
    """Drafts for a batch of histories: (draft_lens [B], drafts [B, gamma_max], -1 padded)."""
    from . import SdvError
    B = len(histories)
    offsets = np.zeros(B + 1, dtype=np.int64)
    for b, h in enumerate(histories):
        offsets[b + 1] = offsets[b] + len(h)
    tokens = np.ascontiguousarray(np.concatenate([np.asarray(h, dtype=np.int32) for h in histories])
                                  if B else np.zeros(0, np.int32), dtype=np.int32)
    lens = np.zeros(B, dtype=np.int32)
    drafts = np.zeros((B, max(gamma_max, 1)), dtype=np.int32)
    rc = load_library().sdv_ngram_draft_batch(_ip(tokens), offsets.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
                                              B, int(min_n), int(max_n), int(gamma_max), _ip(lens), _ip(drafts))
    if rc != SDV_OK:
        raise SdvError(rc, "sdv_ngram_draft_batch")
    return lens, drafts[:, :gamma_max]
