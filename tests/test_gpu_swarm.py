"""The continuous-batching swarm (int4 layer, turnover, compaction, slot
realignment, ragged KV pages) through the C ABI.

* A tiny swarm is compared with the oracle at every step: the oracle carries
  the state (its own K/V rows, lengths, pages, free stack, refills) and each
  step's inputs come from that state and the seeded generators only.
* The 128-slot 9B-class int4 swarm at full size (contexts 1k..16k, gamma by
  the (512 - B) / B rule, so 512 verify rows) is compared with the oracle on
  sampled slots of its first step, then run with turnover on the GPU's own
  state with the invariants checked after every step.
"""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh
from tests import swarm as sw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny_int4_swarm_engine():
    import torch
    assert torch.cuda.is_available()
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 9, fmt="int4")
    eng = gh.engine_for(wl.TINY, 3, wd.weights_to_device(W), max_rows=128, max_slots=32, fmt="int4")
    return W, eng


def test_swarm_tiny_against_oracle_every_step(tiny_int4_swarm_engine):
    W, eng = tiny_int4_swarm_engine
    s = sw.OracleSwarm(wl.TINY, 3, B=24, pool_pages=24 * 25 + 48, ctx=(1, 300), limits=(4, 40), budget=96)
    finished = judged = 0
    for step in range(24):
        batch = s.batch()
        pt_before = batch.page_table.copy()
        status, res, dev = gh.run_step(eng, batch)
        assert status == 0, f"step {step}: status {status}"
        ref = o.verify_step(batch, W)
        fw = ref["forward"]
        p_valid, _ = gh.compare_step(batch, W, fw, res["logits"], res["probs"])
        gh.check_kv_written(batch, fw, dev["kv_pool"], pt_before)
        judged += gh.check_acceptance(batch, p_valid, res["accepted"], res["final_tokens"])
        # realignment from the GPU's own counts, bit-exact, at every step
        gh.check_realign(batch, res, dev)
        finished += s.advance(batch, ref)
    assert finished >= 10, finished          # slots turned over
    # slots whose count or token differs from the oracle's (each within its margin): at most 5 %
    assert judged <= 24 * 24 // 20, judged


def test_swarm_full_size_int4(nine_b_int4):
    from workloads import device as wd
    W, Wd = nine_b_int4
    B, gmax = 128, 3
    eng = gh.engine_for(wl.NINE_B, gmax, Wd, max_rows=512, max_slots=B, fmt="int4")
    pool_pages = B * 1084 + 512
    d = sw.DeviceSwarm(eng, wl.NINE_B, gmax, B, pool_pages, ctx=(1024, 16384), limits=(40, 900), budget=512)
    bd = d.inputs()
    assert bd["R"] == 512 and bd["G"] == 384
    slots = [0, 41, 86, 127]
    sub, rows, pages = sw.host_sub_batch(bd, slots, wl.NINE_B, gmax)
    res = wd.alloc_result(B, bd["R"], wl.NINE_B["vocab"], gmax, d.max_pages, logits=True, probs=True)
    res, acc = d.step(bd, res)
    ref = o.verify_step(sub, W)
    fw = ref["forward"]
    z = res["logits"].cpu().numpy()[rows]
    p = res["probs"].cpu().numpy()[rows]
    p_valid, explained = gh.compare_step(sub, W, fw, z, p)
    assert explained == {}
    gh.check_kv_written(sub, fw, sw.read_pages(bd["kv_pool"], pages), sub.page_table)
    fin = res["final_tokens"].cpu().numpy()
    gh.check_acceptance(sub, p_valid, acc[slots], fin[slots])
    del res, bd
    for _ in range(40):
        d.step()
    assert d.finished_total > 0
