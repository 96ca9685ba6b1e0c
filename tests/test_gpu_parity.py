"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact where the work is integer or the pages' rule decides on given
probabilities (acceptance counts, emitted tokens, page tables, free stack);
within the stated tolerances for the bf16 forward (logits within
1e-2 * rms(logits), probabilities within 1e-3 absolute).
"""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available()
    return torch


# ---------------------------------------------------------------------------
# weight-streaming GEMM (fp32 output, no rounding)
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny_engine(torch_cuda):
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1)
    Wd = wd.weights_to_device(W)
    eng = gh.engine_for(wl.TINY, 3, Wd, max_rows=160, max_slots=16)
    return W, Wd, eng


@pytest.mark.parametrize("xfmt", ["bf16", "f32"])
@pytest.mark.parametrize("rows", [1, 5, 16, 17, 40, 64, 100, 160])
@pytest.mark.parametrize("which", [0, 1, 2, 3, 4, 5])
def test_linear_tiny(tiny_engine, rows, which, xfmt):
    import torch
    W, _, eng = tiny_engine
    names = ["qkv", "o", "gate", "up", "down", None]
    w = W.proj[names[which]] if names[which] else W.w_lm
    K = w.shape[1]
    g = np.random.default_rng(rows * 10 + which)
    x32 = g.standard_normal((rows, K)).astype(np.float32)
    if xfmt == "bf16":
        x = wl.f32_to_bf16_bits(x32)
        xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
        xf = o.bf16_to_f64(x)
    else:
        xd = torch.from_numpy(x32).cuda()
        xf = x32.astype(np.float64)
    y = torch.empty((rows, w.shape[0]), dtype=torch.float32, device="cuda")
    eng.linear(which, xd, y)
    torch.cuda.synchronize()
    ref = o.linear(xf, w)
    err = np.abs(y.cpu().numpy() - ref).max()
    # fp32 accumulation of K exact bf16 products (relative error ~1e-6 of the
    # scale); an fp32 operand enters as bf16 hi + lo (2^-17 relative per value)
    scale = np.sqrt((xf ** 2).sum(1)).max() * np.abs(o.bf16_to_f64(w)).max()
    tol = 1e-5 if xfmt == "bf16" else 3e-5
    assert err <= tol * scale + 1e-6, (err, scale)


@pytest.mark.parametrize("rows", [8, 24, 64])
def test_linear_lm_head_full_size_sampled(nine_b_weights, rows):
    """LM head at full size (151936 x 4096): sampled output columns against float64 dots."""
    import torch
    W, Wd = nine_b_weights
    eng = gh.engine_for(wl.NINE_B, 7, Wd, max_rows=64, max_slots=8)
    g = np.random.default_rng(rows)
    x = wl.f32_to_bf16_bits(g.standard_normal((rows, 4096)).astype(np.float32))
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty((rows, wl.NINE_B["vocab"]), dtype=torch.float32, device="cuda")
    eng.linear(5, xd, y)
    torch.cuda.synchronize()
    cols = np.sort(g.choice(wl.NINE_B["vocab"], size=3000, replace=False))
    cols = np.concatenate([cols, [0, 127, 128, wl.NINE_B["vocab"] - 1]])
    ref = o.bf16_to_f64(x) @ o.bf16_to_f64(W.w_lm[cols]).T
    got = y.cpu().numpy()[:, cols]
    scale = np.abs(ref).max()
    assert np.abs(got - ref).max() <= 2e-5 * scale


# ---------------------------------------------------------------------------
# attention over the paged cache
# ---------------------------------------------------------------------------

def _attention_case(dims, seq_lens, draft_lens, gamma_max, workload, torch):
    from workloads import device as wd
    b = wl.make_batch(dims, workload, seq_lens=seq_lens, draft_lens=draft_lens, gamma_max=gamma_max,
                      extra_pages=2)
    R, nq, D = b.R, dims["n_q"], dims["head_dim"]
    q = np.random.default_rng(workload).standard_normal((R, nq, D)).astype(np.float32)
    bd = wd.batch_to_device(b)
    qd = torch.from_numpy(q).cuda()
    out = torch.zeros((R, nq * D), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    return b, q, bd, qd, out, st


def _attention_ref(dims, b, q):
    nq, nkv, D, P = dims["n_q"], dims["n_kv"], dims["head_dim"], dims["page"]
    pool = o.bf16_to_f64(b.kv_pool)
    qf = q.astype(np.float64)
    offs = wl.row_offsets(b.draft_lens)
    ref = np.zeros((b.R, nq * D))
    for s in range(b.B):
        L, g = int(b.seq_lens[s]), int(b.draft_lens[s])
        Kc, Vc = o.gather_kv(pool, b.page_table[s], L + g + 1, P)
        for i in range(g + 1):
            r = int(offs[s]) + i
            for h in range(nq):
                kv = h // (nq // nkv)
                ref[r, h * D:(h + 1) * D] = o.attention_one(qf[r, h], Kc[kv, :L + i + 1], Vc[kv, :L + i + 1])
    return ref


@pytest.mark.parametrize("case", [
    (wl.TINY, [0, 37, 128, 5], [3, 0, 2, 1], 3),
    (wl.TINY, [300, 16, 15, 1000], [3, 3, 3, 0], 3),
    (wl.NINE_B, [2048], [7], 7),
    (wl.NINE_B, [513, 8000, 1, 4096, 77, 2047, 12000, 640], [3, 1, 2, 0, 3, 2, 1, 3], 3),
    (wl.NINE_B, [16000, 0, 15, 16, 17, 127, 128, 129], [3, 0, 3, 1, 2, 3, 0, 1], 3),
    (wl.NINE_B, [int(x) for x in np.random.default_rng(77).integers(0, 3000, size=40)],
     [int(x) for x in np.random.default_rng(78).integers(0, 4, size=40)], 3),
    # gamma 8: 9 rows x 4 query heads per KV head = 36 query vectors per item
    # (the tcgen05 kernel's 48-vector items)
    (wl.NINE_B, [2048, 2048, 100, 0, 777, 2047, 16, 1500], [8, 8, 8, 8, 0, 5, 8, 3], 8),
    # gamma 11: 48 query vectors, the most one item holds; a long context cut into chunks
    (wl.NINE_B, [3000, 0, 47, 2048, 130, 6000], [11, 11, 4, 9, 11, 0], 11),
    # gamma 15: 64 query vectors, two full items; long contexts split into chunks too
    (wl.NINE_B, [9000, 2048, 0, 5000, 31], [15, 15, 15, 7, 12], 15),
])
@pytest.mark.parametrize("path", [1, 2])
def test_attention_matches_oracle(torch_cuda, case, path):
    """Both attention kernels (1: mma.sync, 2: tcgen05 for head_dim 128) against
    the float64 definition, over ragged lengths, split sequences and partial blocks."""
    dims, lens, gams, gmax = case
    if path == 2 and dims["head_dim"] != 128:
        pytest.skip("the tcgen05 kernel serves head_dim 128")
    torch = torch_cuda
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1) if dims is wl.TINY else None
    # a context only needs the config for attention; weights of the tiny model serve as placeholders
    Wsmall = wd.weights_to_device(W if W is not None else wl.make_weights(wl.TINY, 1))
    cfg = wd.config(dims, gmax)
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine
    if dims is wl.TINY:
        eng = VerifyEngine(cfg, Wsmall, max_rows=64, max_slots=16)
    else:
        eng = _attn_only_engine(cfg, torch)
    eng.set_attention_path(path)
    b, q, bd, qd, out, st = _attention_case(dims, lens, gams, gmax, 40 + len(lens), torch)
    if path == 1 and (gmax + 1) * (dims["n_q"] // dims["n_kv"]) > 48:
        # more query vectors per KV head than the mma.sync kernel holds: refused on the host
        from speculative_decoding_verify_ragged_gb300 import SdvError
        with pytest.raises(SdvError, match="UNSUPPORTED"):
            eng.attention(qd, bd, out, st)
        return
    eng.attention(qd, bd, out, st)
    assert eng.read_status(st) == 0
    got = out.cpu().numpy()
    ref = _attention_ref(dims, b, q)
    err = np.abs(got - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    # q and the softmax weights enter the MMAs as bf16 hi + lo pairs (2^-17
    # relative each), accumulation in fp32: ~1e-5 of the scale
    assert err.max() <= 1e-3 * rms + 1e-4 * np.abs(ref).max(), (err.max(), rms)
    assert np.mean(err) <= 1e-4 * rms


def _attn_only_engine(cfg, torch):
    """A 9B-shaped context whose weight pointers are dummies (attention reads none)."""
    from speculative_decoding_verify_ragged_gb300 import VerifyEngine
    H, V = cfg["hidden"], cfg["vocab"]
    F = cfg["ffn"]
    qd = cfg["n_q"] * cfg["head_dim"]
    nqkv = (cfg["n_q"] + 2 * cfg["n_kv"]) * cfg["head_dim"]
    z = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    Wd = dict(emb=z(8, H), w_qkv=z(nqkv, H), w_o=z(H, qd), w_gate=z(F, H), w_up=z(F, H), w_down=z(H, F),
              w_lm=z(V, H), g_attn=z(H), g_ffn=z(H), g_final=z(H))
    return VerifyEngine(cfg, Wd, max_rows=192, max_slots=48)


# ---------------------------------------------------------------------------
# acceptance + realignment on given probabilities: bit-exact
# ---------------------------------------------------------------------------

def _accept_case(dims, B, gamma_max, seed, finish=True):
    g = np.random.default_rng(seed)
    V = dims["vocab"]
    gam = g.integers(0, gamma_max + 1, size=B)
    lens = g.integers(0, 300, size=B)
    limits = None
    counts = None
    if finish:
        counts = g.integers(0, 40, size=B)
        limits = counts + g.integers(1, gamma_max + 3, size=B)
    b = wl.make_batch(dims, 900 + seed, seq_lens=lens, draft_lens=gam, gamma_max=gamma_max,
                      extra_pages=3 * B, kv_fill="lazy", gen_counts=counts, gen_limits=limits)
    R, G = b.R, b.G
    p = wl.softmax_f32(g.standard_normal((R, V)).astype(np.float32) * 2)
    q = b.draft_probs.copy()
    roff = wl.row_offsets(b.draft_lens)
    goff = np.concatenate([[0], np.cumsum(b.draft_lens)])
    for s in range(B):
        for i in range(int(gam[s])):
            r = int(roff[s]) + i
            x = int(b.tokens[r + 1])
            kind = (s + i) % 5
            if kind == 0:
                q[goff[s] + i] = p[r]                     # q = p: accepted
            elif kind == 1:
                p[r, x] = 0.0                             # the target never writes x: rejected
            elif kind == 2:
                q[goff[s] + i, x] = p[r, x] * 0.5         # p > q at x: accepted
    # a row where max(0, p - q) has no mass: q dominates p everywhere
    if B > 1 and gam[1] > 0:
        r = int(roff[1])
        q[goff[1]] = p[r] * 1.5
        p[r, int(b.tokens[r + 1])] = 0.0
    b.draft_probs = q
    return b, p


# a vocabulary that is not a multiple of 4 (rows not 16-byte aligned: the
# sampling kernel's scalar loads) ending in a partial 512-entry chunk
ODD_VOCAB = dict(wl.TINY, vocab=1003)


@pytest.mark.parametrize("dims,B,gmax,seed", [
    (wl.TINY, 2, 3, 0), (wl.TINY, 17, 3, 1), (wl.TINY, 128, 8, 2),
    (wl.NINE_B, 8, 7, 3), (wl.NINE_B, 3, 3, 4), (ODD_VOCAB, 9, 4, 5),
])
def test_accept_and_realign_bit_exact(torch_cuda, dims, B, gmax, seed):
    import torch
    from workloads import device as wd
    b, p = _accept_case(dims, B, gmax, seed)
    eng = _attn_only_engine(wd.config(dims, gmax), torch) if dims is not wl.TINY else \
        gh.engine_for(dims, gmax, wd.weights_to_device(wl.make_weights(wl.TINY, 1)), max(b.R, 16), 256)
    bd = wd.batch_to_device(b)
    res = wd.alloc_result(b.B, b.R, dims["vocab"], gmax, b.page_table.shape[1])
    pd = torch.from_numpy(p).cuda()
    eng.accept(pd, bd, res)
    assert eng.read_status(res["status"]) == 0
    acc, emitted, eoff, fin = o.accept_batch(p, b.draft_probs, b.tokens, b.uniforms, b.draft_lens)
    ra = o.realign(b.seq_lens, acc, b.page_table, b.num_pages, b.free_pages, b.num_free, dims["page"], gmax,
                   gen_counts=b.gen_counts, gen_limits=b.gen_limits)
    c = lambda k: res[k].cpu().numpy()  # noqa: E731
    assert np.array_equal(c("accepted"), acc)
    assert np.array_equal(c("final_tokens"), fin)
    assert np.array_equal(c("emitted_offsets"), eoff)
    assert np.array_equal(c("emitted_tokens")[:eoff[-1]], emitted)
    assert np.array_equal(c("new_seq_lens"), ra["new_seq_lens"])
    assert np.array_equal(c("finished"), ra["finished"])
    assert ra["status"] == 0
    assert np.array_equal(bd["page_table"].cpu().numpy(), ra["page_table"])
    assert np.array_equal(bd["num_pages"].cpu().numpy(), ra["num_pages"])
    nf = int(bd["num_free_out"].cpu().numpy()[0])
    assert nf == ra["num_free"]
    assert np.array_equal(bd["free_pages"].cpu().numpy()[:nf], ra["free_pages"][:nf])
    nl = int(c("num_live")[0])
    assert nl == ra["num_live"]
    assert np.array_equal(c("next_src")[:nl], ra["next_src"])
    assert np.array_equal(c("next_seq_lens")[:nl], ra["next_seq_lens"])
    assert np.array_equal(c("next_page_table")[:nl], ra["next_page_table"])
    assert np.array_equal(c("next_gen_counts")[:nl], ra["next_gen_counts"])
    tested, accepted = o.accept_histogram(acc, b.draft_lens, gmax)
    assert np.array_equal(c("accept_tested")[:gmax], tested)
    assert np.array_equal(c("accept_accepted")[:gmax], accepted)


# ---------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------

def _full_step_check(eng, W, batch, name):
    pt_before = batch.page_table.copy()
    status, res, dev = gh.run_step(eng, batch)
    assert status == 0, f"{name}: status {status}"
    ref = o.verify_step(batch, W)
    fw = ref["forward"]
    # every row inside the tolerance (9B-class layer: as computed, no other roundings)
    p_valid, explained = gh.compare_step(batch, W, fw, res["logits"], res["probs"])
    if not gh.flips_allowed(batch.dims):
        assert explained == {}
    # every row's K/V landed in its page at position L + i, rounded as the oracle
    # rounds it (or, within the window, to the other neighbour)
    gh.check_kv_written(batch, fw, dev["kv_pool"], pt_before)
    judged = gh.check_acceptance(batch, p_valid, res["accepted"], res["final_tokens"])
    # realignment from the GPU's counts, bit-exact, whether or not they equal the oracle's
    gh.check_realign(batch, res, dev)
    return judged


def test_step_tiny_workload(tiny_engine):
    W, _, eng = tiny_engine
    for variant in range(3):
        if variant == 0:
            batch = wl.workload1()
        elif variant == 1:
            batch = wl.make_batch(wl.TINY, 11, seq_lens=[0, 37, 128, 5, 200], draft_lens=[3, 0, 2, 1, 3],
                                  gamma_max=3, extra_pages=6)
        else:
            batch = wl.make_batch(wl.TINY, 12, seq_lens=list(range(1, 34, 4)), draft_lens=[3, 2, 1, 0, 3, 2, 1, 0, 3],
                                  gamma_max=3, extra_pages=12, gen_counts=[0] * 9,
                                  gen_limits=[1, 2, 3, 4, 5, 100, 100, 100, 2])
        _full_step_check(eng, W, batch, f"tiny{variant}")


@pytest.fixture(scope="module")
def nine_b_engine(nine_b_weights):
    W, Wd = nine_b_weights
    return W, gh.engine_for(wl.NINE_B, 7, Wd, max_rows=64, max_slots=16)


def _retargeted(batch, W, workload):
    fw = o.forward(batch.dims, W, batch.kv_pool, batch.page_table, batch.seq_lens, batch.draft_lens,
                   batch.tokens)
    wl.retarget_draft_probs(batch, fw["probs"].astype(np.float32), workload)
    return batch


def test_step_batch_of_one(nine_b_engine):
    """B = 1, gamma = 7, 9B-class layer, ctx 2048, acceptance 0.8."""
    W, eng = nine_b_engine
    batch = _retargeted(wl.workload2(), W, 2)
    _full_step_check(eng, W, batch, "workload2")


def test_step_eight_agents(nine_b_engine):
    """B = 8 ragged, gamma_b in {1,2,3}, ctx 512..8192, acceptance {0.97, 0.8, 0.14}."""
    W, eng = nine_b_engine
    lens, gam, alphas = wl.workload3_shape()
    batch = wl.make_batch(wl.NINE_B, 3, seq_lens=lens, draft_lens=gam, gamma_max=7, alphas=alphas,
                          extra_pages=16)
    batch = _retargeted(batch, W, 3)
    _full_step_check(eng, W, batch, "workload3")


def test_step_batch_equivalence(tiny_engine):
    """A sequence's logits are the same alone and inside the ragged batch (and permuted)."""
    W, _, eng = tiny_engine
    batch = wl.make_batch(wl.TINY, 21, seq_lens=[5, 90, 33, 0], draft_lens=[2, 3, 0, 1], gamma_max=3,
                          extra_pages=4)
    _, full, _ = gh.run_step(eng, batch)
    offs = wl.row_offsets(batch.draft_lens)
    for s in range(batch.B):
        one = wl.Batch(dims=batch.dims, gamma_max=3, seq_lens=batch.seq_lens[s:s + 1],
                       draft_lens=batch.draft_lens[s:s + 1], tokens=batch.tokens[offs[s]:offs[s + 1]],
                       draft_probs=batch.draft_probs[int(offs[s]) - s:int(offs[s + 1]) - s - 1],
                       uniforms=batch.uniforms[offs[s]:offs[s + 1]], kv_pool=batch.kv_pool,
                       page_table=batch.page_table[s:s + 1], num_pages=batch.num_pages[s:s + 1],
                       free_pages=batch.free_pages, num_free=batch.num_free)
        _, alone, _ = gh.run_step(eng, one)
        a, b_ = alone["logits"], full["logits"][offs[s]:offs[s + 1]]
        # the same rows through a different split of the attention work: equal up to
        # a rare one-ulp bf16 flip of an intermediate
        assert np.max(np.abs(a - b_)) <= 2e-3 * np.sqrt(np.mean(b_ ** 2))


# ---------------------------------------------------------------------------
# device-detected errors: status word, no trap, context still usable
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fault", ["token", "gamma", "page", "cover", "rows", "capacity"])
def test_device_errors_set_status(tiny_engine, fault):
    import torch
    from workloads import device as wd
    W, _, eng = tiny_engine
    batch = wl.workload1()
    if fault == "capacity":
        # pages cover this step but the realigned length needs one more, and none are free
        batch = wl.make_batch(wl.TINY, 1, seq_lens=[124, 124], draft_lens=[3, 1], gamma_max=3, extra_pages=0)
    if fault == "token":
        batch.tokens[2] = batch.dims["vocab"] + 5
    elif fault == "page":
        batch.page_table[0, 1] = batch.kv_pool.shape[0] + 3
    elif fault == "cover":
        batch.num_pages[0] = 1
    bd = wd.batch_to_device(batch)
    if fault == "gamma":
        bd["draft_lens"][1] = 9          # beyond gamma_max = 3
    if fault == "rows":
        # claim one row more than the draft lengths give (buffers padded so nothing reads past them)
        bd["R"] = bd["R"] + 1
        bd["G"] = bd["G"] + 1
        bd["tokens"] = torch.cat([bd["tokens"], torch.zeros(1, dtype=torch.int32, device="cuda")])
        bd["uniforms"] = torch.cat([bd["uniforms"], torch.zeros(1, dtype=torch.float32, device="cuda")])
    res = wd.alloc_result(batch.B, batch.R + 1, batch.dims["vocab"], 3, batch.page_table.shape[1])
    eng.verify_step(bd, res)
    st = eng.read_status(res["status"])
    expect = {"token": 6, "gamma": 6, "page": 3, "cover": 3, "rows": 6, "capacity": 2}[fault]
    assert st == expect, (fault, st)
    # the context is still usable
    ok = wl.workload1()
    status, _, _ = gh.run_step(eng, ok)
    assert status == 0


# ---------------------------------------------------------------------------
# a failed call leaves the context ready for the next one
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dims", [wl.TINY, wl.NINE_B])
def test_call_after_a_zero_mass_row_is_bit_exact(torch_cuda, dims):
    """A batch whose bonus row has no probability mass sets SDV_ERR_BAD_INPUT
    from inside the sampling kernel while the other sequences' blocks still
    run; the valid call that follows on the same context must be bit-exact
    with the oracle (every sequence's sampling arrival counter back at zero)."""
    import torch
    from workloads import device as wd
    gmax = 3
    eng = _attn_only_engine(wd.config(dims, gmax), torch) if dims is not wl.TINY else \
        gh.engine_for(dims, gmax, wd.weights_to_device(wl.make_weights(wl.TINY, 1)), 256, 64)
    for rep in range(3):
        b, p = _accept_case(dims, 48, gmax, 40 + rep, finish=False)
        # slot 5 drafts nothing; its only row (the bonus distribution) is all zeros
        bad = wl.make_batch(dims, 940 + rep, seq_lens=b.seq_lens, draft_lens=np.where(np.arange(48) == 5, 0,
                                                                                           b.draft_lens),
                            gamma_max=gmax, extra_pages=3 * 48, kv_fill="lazy")
        pbad = wl.softmax_f32(np.random.default_rng(rep).standard_normal((bad.R, dims["vocab"])).astype(np.float32))
        pbad[int(wl.row_offsets(bad.draft_lens)[5])] = 0.0
        bdb = wd.batch_to_device(bad)
        rb = wd.alloc_result(bad.B, bad.R, dims["vocab"], gmax, bad.page_table.shape[1])
        eng.accept(torch.from_numpy(pbad).cuda(), bdb, rb)
        assert eng.read_status(rb["status"]) == 6
        # the valid call on the same context
        bd = wd.batch_to_device(b)
        res = wd.alloc_result(b.B, b.R, dims["vocab"], gmax, b.page_table.shape[1])
        eng.accept(torch.from_numpy(p).cuda(), bd, res)
        assert eng.read_status(res["status"]) == 0
        acc, emitted, eoff, fin = o.accept_batch(p, b.draft_probs, b.tokens, b.uniforms, b.draft_lens)
        assert np.array_equal(res["accepted"].cpu().numpy(), acc)
        assert np.array_equal(res["final_tokens"].cpu().numpy(), fin)
        assert np.array_equal(res["emitted_tokens"].cpu().numpy()[:eoff[-1]], emitted)


@pytest.mark.parametrize("fault", ["negative", "beyond_gamma", "token"])
def test_realign_rejects_bad_counts_and_writes_nothing(tiny_engine, fault):
    """sdv_realign takes the accepted counts and final tokens from the caller:
    a count outside 0..gamma_b or a token outside the vocabulary is
    SDV_ERR_BAD_INPUT, and no output, page or free-stack entry moves."""
    import torch
    from workloads import device as wd
    _, _, eng = tiny_engine
    b = wl.make_batch(wl.TINY, 77, seq_lens=[30, 60, 5], draft_lens=[3, 2, 1], gamma_max=3, extra_pages=6)
    acc = np.array([1, 2, 0], np.int32)
    fin = np.array([7, 8, 9], np.int32)
    if fault == "negative":
        acc[1] = -1
    elif fault == "beyond_gamma":
        acc[2] = 2          # gamma of slot 2 is 1
    else:
        fin[0] = wl.TINY["vocab"]
    bd = wd.batch_to_device(b)
    res = wd.alloc_result(b.B, b.R, wl.TINY["vocab"], 3, b.page_table.shape[1])
    res["accepted"].copy_(torch.from_numpy(acc))
    res["final_tokens"].copy_(torch.from_numpy(fin))
    sentinel = -12345
    for k in ("emitted_tokens", "emitted_offsets", "new_seq_lens", "finished", "next_src", "next_seq_lens"):
        res[k].fill_(sentinel)
    eng.realign(bd, res)
    assert eng.read_status(res["status"]) == 6
    for k in ("emitted_tokens", "emitted_offsets", "new_seq_lens", "finished", "next_src", "next_seq_lens"):
        assert (res[k].cpu().numpy() == sentinel).all(), k
    assert np.array_equal(bd["page_table"].cpu().numpy(), b.page_table)
    assert np.array_equal(bd["num_pages"].cpu().numpy(), b.num_pages)
    assert int(bd["num_free_out"].cpu().numpy()[0]) == b.num_free
    assert np.array_equal(bd["free_pages"].cpu().numpy(), b.free_pages)


def test_bounded_wait_times_out_and_the_context_recovers(tiny_engine):
    """The device timeout path: with the test hook set, the step's first kernel
    waits on a barrier nothing completes, gives up after 2 ms and records
    SDV_ERR_TIMEOUT; no output is written; the next step on the same context,
    hook off, returns SDV_OK and matches the oracle."""
    import torch
    from workloads import device as wd
    W, _, eng = tiny_engine
    batch = wl.workload1()
    bd = wd.batch_to_device(batch)
    res = wd.alloc_result(batch.B, batch.R, batch.dims["vocab"], 3, batch.page_table.shape[1], logits=True)
    res["accepted"].fill_(-7)
    res["logits"].fill_(-7.0)
    eng.set_stall_test(2_000_000)
    try:
        eng.verify_step(bd, res)
        assert eng.read_status(res["status"]) == 5          # SDV_ERR_TIMEOUT
    finally:
        eng.set_stall_test(0)
    assert (res["accepted"].cpu().numpy() == -7).all()
    assert (res["logits"].cpu().numpy() == -7.0).all()
    assert np.array_equal(bd["page_table"].cpu().numpy(), batch.page_table)
    _full_step_check(eng, W, wl.workload1(), "after-timeout")
