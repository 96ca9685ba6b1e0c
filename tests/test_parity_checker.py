"""The comparison the GPU step tests use, exercised on the CPU with results
made by the oracle itself: on the tiny model, ONE valid alternative rounding
of a value at a bf16 tie passes, a planted logit error of the same size does
not, and on the 9B-class layer no alternative rounding is tried at all.

The case is a wide tiny-model batch in which V element 36 of head 0 in row 0
(a one-token sequence at position 0) lies 6.4e-7 relative from a bf16 tie;
its other rounding moves that row's logits by 1.13 % of their rms, more than
the 1 % tolerance, so only the tie-aware path can accept it.
"""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh


@pytest.fixture(autouse=True)
def _uncounted():
    """The checker's own tests plant their roundings: keep them out of the
    session's count of roundings the GPU comparisons used."""
    saved = list(gh.FLIPS_USED)
    yield
    gh.FLIPS_USED[:] = saved


@pytest.fixture(scope="module")
def wide():
    W = wl.make_weights(wl.TINY, 1)
    lens = list(range(0, 400, 7))[:57]
    gam = [(3 * i) % 4 for i in range(57)]
    batch = wl.make_batch(wl.TINY, 31, seq_lens=lens, draft_lens=gam, gamma_max=3, extra_pages=80)
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens,
                   batch.tokens)
    return W, batch, fw


def _noise(z, seed):
    return z + 1e-4 * np.sqrt(np.mean(z ** 2)) * np.random.default_rng(seed).standard_normal(z.shape)


def test_exact_result_needs_no_explanation(wide):
    W, batch, fw = wide
    p, ex = gh.compare_step(batch, W, fw, _noise(fw["logits"], 0).astype(np.float32),
                            fw["probs"].astype(np.float32))
    assert ex == {} and np.array_equal(p, fw["probs"])


def test_other_rounding_at_a_tie_is_accepted(wide):
    W, batch, fw = wide
    d, _, _ = gh._tie_distance(fw["v_pre"][0], axis=1)
    assert d[0, 36] < gh.TIE_WINDOW
    alt = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens,
                    batch.tokens, flips={("v", 0, 0, 36)})
    rms = np.sqrt(np.mean(fw["logits"] ** 2))
    assert np.abs(alt["logits"][0] - fw["logits"][0]).max() > gh.LOGIT_TOL_REL_RMS * rms
    p, ex = gh.compare_step(batch, W, fw, _noise(alt["logits"], 1).astype(np.float32),
                            alt["probs"].astype(np.float32))
    assert ex == {0: ("v", 0, 0, 36)}
    assert np.array_equal(p[0], alt["probs"][0])


def test_planted_error_is_rejected(wide):
    W, batch, fw = wide
    z = fw["logits"].copy()
    rms = np.sqrt(np.mean(z ** 2))
    z[5, 17] += 1.2 * gh.LOGIT_TOL_REL_RMS * rms
    with pytest.raises(AssertionError):
        gh.compare_step(batch, W, fw, z.astype(np.float32), None)


def test_kv_check_rejects_a_far_rounding(wide):
    """K/V in the pool: the oracle's rounding passes, the other neighbour only inside the window."""
    W, batch, fw = wide
    pool = batch.kv_pool.copy()
    P = batch.dims["page"]
    offs = wl.row_offsets(batch.draft_lens)
    for (b, pos), (k, v) in fw["kv_rows"].items():
        pg = batch.page_table[b, pos // P]
        pool[pg, :, 0, pos % P, :] = o.f64_to_bf16_bits(k)
        pool[pg, :, 1, pos % P, :] = o.f64_to_bf16_bits(v)
    assert gh.check_kv_written(batch, fw, pool, batch.page_table) == 0
    # the tie at row 0, v head 0, element 36 may take the other neighbour
    pg = batch.page_table[0, 0]
    ok = pool.copy()
    ok[pg, 0, 1, 0, 36] = o.f64_to_bf16_bits(o.round_bf16_other(fw["v_pre"][0, 0, 36], fw["kv_rows"][(0, 0)][1][0, 36]))
    assert gh.check_kv_written(batch, fw, ok, batch.page_table) == 1
    # a value far from any tie may not
    d, near, far = gh._tie_distance(fw["v_pre"][0], axis=1)
    j = int(np.argmax(np.where(np.isfinite(d[1]), d[1], -1)))
    bad = pool.copy()
    bad[pg, 1, 1, 0, j] = o.f64_to_bf16_bits(far[1, j:j + 1])[0]
    with pytest.raises(AssertionError):
        gh.check_kv_written(batch, fw, bad, batch.page_table)
    del offs


def test_nine_b_rows_get_no_other_rounding(wide):
    """The same result, presented as a 9B-class batch: the row outside the
    tolerance fails outright (the checker tries no other rounding there)."""
    import dataclasses
    W, batch, fw = wide
    alt = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens,
                    batch.tokens, flips={("v", 0, 0, 36)})
    big = dataclasses.replace(batch, dims=dict(batch.dims, hidden=4096))
    assert not gh.flips_allowed(big.dims)
    with pytest.raises(AssertionError, match="outside tolerance"):
        gh.compare_step(big, W, fw, alt["logits"].astype(np.float32), alt["probs"].astype(np.float32))


def test_tie_window_is_the_measured_error():
    """A candidate for another rounding must lie within 2^-17 rms of a tie (the
    largest error seen on the GPU), not a multiple of it."""
    assert gh.TIE_WINDOW == 2.0 ** -17
    assert gh.KV_WINDOW <= 2.0 ** -15
