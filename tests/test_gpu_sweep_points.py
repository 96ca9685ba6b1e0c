"""The crossover sweep's largest points (9B-class layer, bf16, context 2048)
against the oracle, through the C ABI, in the launch configuration the bench
times: B = 128 with gamma = 3 (512 verify rows, tcgen05 GEMMs and attention),
B = 64 with gamma = 8 (576 rows: 36 query vectors per KV head, the mma.sync
attention kernel) and B = 128 with gamma = 8 (1152 rows, a ragged last
256-row activation tile in the LM head).

The GPU runs the whole batch; the oracle recomputes a sample of its sequences
one by one (each sequence's rows depend only on its own cache, so a subset is
exact).  The sampled sequences' draft distributions are rebuilt around the
oracle's own target probabilities (per-draft acceptance 0.8); the others keep
the recipe's q.  Checked: logits and probabilities of every sampled row within
the stated tolerances with no other rounding allowed, their K/V rows in the
pages, their acceptance counts and final tokens, and the realignment of the
whole batch from the GPU's counts, bit-exact.  The LM head alone is checked on
sampled columns at 512, 1024 and 1152 rows on the tcgen05 kernel.
"""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh
from tests import swarm as sw

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,gamma", [(128, 3), (64, 8), (128, 8)])
def test_sweep_point_step_sampled(nine_b_weights, B, gamma):
    import torch
    from workloads import device as wd
    W, Wd = nine_b_weights
    batch = wl.workload4(B, gamma, kv_fill="lazy", extra_pages=4 * B + 8)
    eng = gh.engine_for(wl.NINE_B, batch.gamma_max, Wd, max_rows=batch.R, max_slots=B)
    bd = wd.batch_to_device(batch)
    wd.normal_bf16_device_(bd["kv_pool"], wl._key(4, wl.S_KV, 1000 * B + gamma))
    slots = [0, 1, B // 2 + 3, B - 1]
    sub, rows, pages = sw.host_sub_batch(bd, slots, wl.NINE_B, batch.gamma_max)
    # the sampled sequences' q rebuilt around the oracle's own p (acceptance 0.8)
    fw0 = o.forward(sub.dims, W, sub.kv_pool, sub.page_table, sub.seq_lens, sub.draft_lens, sub.tokens)
    sub.alphas = np.full(len(slots), 0.8)
    wl.retarget_draft_probs(sub, fw0["probs"].astype(np.float32), 4)
    goff = np.concatenate([[0], np.cumsum(batch.draft_lens)])
    g_rows = np.concatenate([np.arange(goff[s], goff[s + 1]) for s in slots]).astype(np.int64)
    bd["draft_probs"][torch.from_numpy(g_rows).cuda()] = torch.from_numpy(sub.draft_probs).cuda()
    host_before = {k: bd[k].cpu().numpy() for k in ("page_table", "num_pages", "free_pages", "draft_probs")}
    res = wd.alloc_result(B, batch.R, wl.NINE_B["vocab"], batch.gamma_max, batch.page_table.shape[1],
                          logits=True, probs=True)
    eng.verify_step(bd, res)
    assert eng.read_status(res["status"]) == 0
    torch.cuda.synchronize()

    ref = o.verify_step(sub, W)
    fw = ref["forward"]
    z = res["logits"][torch.from_numpy(rows).cuda()].cpu().numpy()
    p = res["probs"][torch.from_numpy(rows).cuda()].cpu().numpy()
    p_valid, explained = gh.compare_step(sub, W, fw, z, p)
    assert explained == {}
    gh.check_kv_written(sub, fw, sw.read_pages(bd["kv_pool"], pages), sub.page_table)
    out = gh.to_numpy({k: v for k, v in res.items() if k not in ("logits", "probs")})
    gh.check_acceptance(sub, p_valid, out["accepted"][slots], out["final_tokens"][slots])
    # the whole batch's realignment from the GPU's counts, bit-exact
    full = wl.Batch(dims=batch.dims, gamma_max=batch.gamma_max, seq_lens=batch.seq_lens,
                    draft_lens=batch.draft_lens, tokens=batch.tokens, draft_probs=host_before["draft_probs"],
                    uniforms=batch.uniforms, kv_pool=np.zeros((0,), np.uint16),
                    page_table=host_before["page_table"], num_pages=host_before["num_pages"],
                    free_pages=host_before["free_pages"], num_free=batch.num_free)
    gh.check_realign(full, out, gh.to_numpy({k: bd[k] for k in ("page_table", "num_pages", "free_pages",
                                                               "num_free_out")}))


@pytest.fixture(scope="module")
def lm_engine(nine_b_weights):
    W, Wd = nine_b_weights
    return W, gh.engine_for(wl.NINE_B, 8, Wd, max_rows=1152, max_slots=128)


@pytest.mark.parametrize("rows", [512, 1024, 1152])
def test_lm_head_large_rows_tcgen05(lm_engine, rows):
    """The 151936 x 4096 LM head at the sweep's row counts on tcgen05: sampled
    columns (the first and last vocabulary tiles included) of every row, the
    ragged last 256-row activation tile among them, against float64 dots."""
    import torch
    W, eng = lm_engine
    g = np.random.default_rng(90 + rows)
    x = wl.f32_to_bf16_bits(g.standard_normal((rows, 4096)).astype(np.float32))
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty((rows, wl.NINE_B["vocab"]), dtype=torch.float32, device="cuda")
    eng.set_gemm_path(2)
    try:
        eng.linear(5, xd, y)
    finally:
        eng.set_gemm_path(0)
    torch.cuda.synchronize()
    cols = np.sort(g.choice(wl.NINE_B["vocab"], size=1500, replace=False))
    cols = np.unique(np.concatenate([cols, [0, 127, 128, wl.NINE_B["vocab"] - 1]]))
    got = y[:, torch.from_numpy(cols).cuda()].cpu().numpy()
    ref = o.bf16_to_f64(x) @ o.bf16_to_f64(W.w_lm[cols]).T
    assert np.abs(got - ref).max() <= 2e-5 * np.abs(ref).max()
