"""sdv_accept_static: the entry point that allocates nothing.

Some callers cannot allocate device memory when they verify drafts (memory
carved up once at start-up, work recorded inside a CUDA-graph capture, a
plugin whose host framework owns every allocation).  sdv_accept_static keeps
its scratch in a static device array instead of a caller-provided workspace.
This test calls it through the C ABI twice in a row and checks each result
against sdv_accept on a context (bit-exact: the same rule on the same
probabilities and uniforms).  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu


def _case(seed):
    g = np.random.default_rng(seed)
    dims = wl.TINY
    B, gmax = 12, 3
    gam = g.integers(0, gmax + 1, size=B)
    lens = g.integers(0, 200, size=B)
    counts = g.integers(0, 30, size=B)
    limits = counts + g.integers(1, gmax + 3, size=B)
    b = wl.make_batch(dims, 700 + seed, seq_lens=lens, draft_lens=gam, gamma_max=gmax, extra_pages=3 * B,
                      kv_fill="lazy", gen_counts=counts, gen_limits=limits)
    p = wl.softmax_f32(g.standard_normal((b.R, dims["vocab"])).astype(np.float32) * 2)
    return b, p, gmax


def _run(fn, b, p, gmax):
    import torch
    from workloads import device as wd
    bd = wd.batch_to_device(b)
    res = wd.alloc_result(b.B, b.R, b.dims["vocab"], gmax, b.page_table.shape[1])
    fn(torch.from_numpy(p).cuda(), bd, res)
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in res.items()}
    out["page_table_after"] = bd["page_table"].cpu().numpy()
    out["free_after"] = bd["free_pages"].cpu().numpy()
    out["num_free_after"] = int(bd["num_free_out"].cpu().numpy()[0])
    return out


def test_accept_static_matches_context_entry_point():
    import torch
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine, _abi
    from workloads import device as wd
    lib = _abi.load_library()
    dims = wl.TINY
    cfg_d = wd.config(dims, 3)
    cfg = VerifyEngine(cfg_d, wd.weights_to_device(wl.make_weights(dims, 1)), max_rows=64, max_slots=16)

    def with_context(probs, bd, res):
        cfg.accept(probs, bd, res)

    def static(probs, bd, res):
        bs = VerifyEngine.batch_struct(bd)
        rs = VerifyEngine.result_struct(res)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lib.sdv_accept_static(ctypes.byref(cfg.cfg), ctypes.c_void_p(probs.data_ptr()), ctypes.byref(bs),
                                   ctypes.byref(rs), stream)
        assert rc == _abi.SDV_OK

    for call, seed in enumerate((1, 2)):        # two calls in a row share the static scratch
        b, p, gmax = _case(seed)
        ref = _run(with_context, b, p, gmax)
        got = _run(static, b, p, gmax)
        assert got["status"][0] == 0 and ref["status"][0] == 0
        for k in ("accepted", "final_tokens", "emitted_offsets", "new_seq_lens", "finished", "new_gen_counts",
                  "num_live", "next_src", "next_seq_lens", "next_num_pages", "next_page_table",
                  "accept_tested", "accept_accepted", "page_table_after"):
            assert np.array_equal(got[k], ref[k]), (call, k)
        n = int(ref["emitted_offsets"][-1])
        assert np.array_equal(got["emitted_tokens"][:n], ref["emitted_tokens"][:n])
        assert got["num_free_after"] == ref["num_free_after"]
        nf = ref["num_free_after"]
        assert np.array_equal(got["free_after"][:nf], ref["free_after"][:nf])


def test_accept_static_rejects_sizes_beyond_its_scratch():
    import torch
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine, _abi
    from workloads import device as wd
    lib = _abi.load_library()
    cfg = wd.config(wl.TINY, 3)
    c = _abi.SdvConfig(*[int(cfg[k]) for k in ("hidden", "n_q", "n_kv", "head_dim", "ffn", "vocab", "page_size",
                                                "gamma_max", "weight_format")], 1e-6, 1e6)
    c.vocab = 262144 + 1
    b, p, gmax = _case(3)
    bd = wd.batch_to_device(b)
    res = wd.alloc_result(b.B, b.R, 1024, gmax, b.page_table.shape[1])
    bs = VerifyEngine.batch_struct(bd)
    rs = VerifyEngine.result_struct(res)
    probs = torch.from_numpy(p).cuda()
    rc = lib.sdv_accept_static(ctypes.byref(c), ctypes.c_void_p(probs.data_ptr()), ctypes.byref(bs),
                               ctypes.byref(rs), None)
    assert rc == _abi.SDV_ERR_CAPACITY


def test_accept_static_full_vocabulary_matches_the_oracle():
    """sdv_accept_static with the 151936-entry vocabulary against the oracle's
    acceptance and realignment, bit-exact: every draft's verdict, the final
    draw (297 sampling chunks per row, the last one partial) and the state the
    realignment writes."""
    import torch
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine, _abi
    from workloads import device as wd
    from oracle import verify_step as o
    lib = _abi.load_library()
    dims, B, gmax = wl.NINE_B, 8, 7
    cfg = wd.config(dims, gmax)
    c = _abi.SdvConfig(*[int(cfg[k]) for k in ("hidden", "n_q", "n_kv", "head_dim", "ffn", "vocab", "page_size",
                                                "gamma_max", "weight_format")], 1e-6, 1e6)
    g = np.random.default_rng(31)
    gam = g.integers(0, gmax + 1, size=B)
    gam[0], gam[1] = 0, gmax                      # a bonus-only slot and a full-length one
    lens = g.integers(0, 300, size=B)
    counts = g.integers(0, 40, size=B)
    limits = counts + g.integers(1, gmax + 3, size=B)
    b = wl.make_batch(dims, 760, seq_lens=lens, draft_lens=gam, gamma_max=gmax, extra_pages=3 * B,
                      kv_fill="lazy", gen_counts=counts, gen_limits=limits)
    p = wl.softmax_f32(g.standard_normal((b.R, dims["vocab"])).astype(np.float32) * 2)
    # half the drafts drawn from a q equal to p (accepted whatever u is)
    roff = wl.row_offsets(b.draft_lens)
    goff = np.concatenate([[0], np.cumsum(b.draft_lens)])
    for s in range(0, B, 2):
        for i in range(int(gam[s])):
            b.draft_probs[goff[s] + i] = p[int(roff[s]) + i]
    bd = wd.batch_to_device(b)
    res = wd.alloc_result(b.B, b.R, dims["vocab"], gmax, b.page_table.shape[1])
    bs = VerifyEngine.batch_struct(bd)
    rs = VerifyEngine.result_struct(res)
    probs = torch.from_numpy(p).cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.sdv_accept_static(ctypes.byref(c), ctypes.c_void_p(probs.data_ptr()), ctypes.byref(bs),
                                 ctypes.byref(rs), stream) == _abi.SDV_OK
    torch.cuda.synchronize()
    acc, emitted, eoff, fin = o.accept_batch(p, b.draft_probs, b.tokens, b.uniforms, b.draft_lens)
    ra = o.realign(b.seq_lens, acc, b.page_table, b.num_pages, b.free_pages, b.num_free, dims["page"], gmax,
                   gen_counts=b.gen_counts, gen_limits=b.gen_limits)
    r = {k: v.cpu().numpy() for k, v in res.items()}
    assert r["status"][0] == 0 and ra["status"] == 0
    assert np.array_equal(r["accepted"], acc)
    assert np.array_equal(r["final_tokens"], fin)
    assert np.array_equal(r["emitted_offsets"], eoff)
    assert np.array_equal(r["emitted_tokens"][:eoff[-1]], emitted)
    assert np.array_equal(r["new_seq_lens"], ra["new_seq_lens"])
    assert np.array_equal(r["finished"], ra["finished"])
    assert np.array_equal(bd["page_table"].cpu().numpy(), ra["page_table"])
    nf = int(bd["num_free_out"].cpu().numpy()[0])
    assert nf == ra["num_free"]
    assert np.array_equal(bd["free_pages"].cpu().numpy()[:nf], ra["free_pages"][:nf])
    nl = int(r["num_live"][0])
    assert nl == ra["num_live"]
    assert np.array_equal(r["next_src"][:nl], ra["next_src"])
    assert np.array_equal(r["next_page_table"][:nl], ra["next_page_table"])
