"""The full-size LM head against float64 dots across the vocabulary (first
tiles, the last eighth, the ragged last tile), and determinism: a tile cut
between CTAs is summed from its pieces in CTA order, so repeated runs of a GEMM
and of a whole step give identical bits."""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu
MMA_SYNC, TCGEN05 = 1, 2


def _lm_head(eng, x, path):
    import torch
    eng.set_gemm_path(path)
    try:
        xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
        y = torch.empty((x.shape[0], wl.NINE_B["vocab"]), dtype=torch.float32, device="cuda")
        eng.linear(5, xd, y)
        torch.cuda.synchronize()
        return y.cpu().numpy()
    finally:
        eng.set_gemm_path(0)


@pytest.mark.parametrize("rows,path", [(1, MMA_SYNC), (8, MMA_SYNC), (13, MMA_SYNC), (16, MMA_SYNC),
                                       (24, TCGEN05), (64, TCGEN05)])
def test_lm_head_columns_and_repeats(nine_b_weights, rows, path):
    """151936 x 4096: columns of the first seven eighths, of the last eighth of
    the 1187 vocabulary tiles and of the ragged last tile against float64;
    three runs give the same bits."""
    W, Wd = nine_b_weights
    eng = gh.engine_for(wl.NINE_B, 7, Wd, max_rows=64, max_slots=8)
    g = np.random.default_rng(70 + rows)
    x = wl.f32_to_bf16_bits(g.standard_normal((rows, 4096)).astype(np.float32))
    ys = [_lm_head(eng, x, path) for _ in range(3)]
    V = wl.NINE_B["vocab"]
    tail0 = (1187 - (1187 + 7) // 8) * 128
    cols = np.concatenate([g.choice(tail0, size=1500, replace=False),
                           tail0 + g.choice(V - tail0, size=1500, replace=False),
                           [0, tail0 - 1, tail0, tail0 + 127, V - 129, V - 128, V - 1]])
    cols = np.unique(cols)
    ref = o.bf16_to_f64(x) @ o.bf16_to_f64(W.w_lm[cols]).T
    assert np.abs(ys[0][:, cols] - ref).max() <= 2e-5 * np.abs(ref).max()
    assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


def test_step_repeats_bit_for_bit(nine_b_weights):
    """The batch-of-one step run three times from the same state: identical
    logits and results."""
    import torch
    from workloads import device as wd
    W, Wd = nine_b_weights
    eng = gh.engine_for(wl.NINE_B, 7, Wd, max_rows=64, max_slots=8)
    batch = wl.workload2(extra_pages=8)
    outs = []
    for _ in range(3):
        bd = wd.batch_to_device(batch)
        res = wd.alloc_result(batch.B, batch.R, wl.NINE_B["vocab"], 7, batch.page_table.shape[1], logits=True)
        eng.verify_step(bd, res)
        assert eng.read_status(res["status"]) == 0
        torch.cuda.synchronize()
        outs.append(gh.to_numpy(res))
    for k in ("logits", "accepted", "final_tokens", "emitted_tokens", "new_seq_lens"):
        assert np.array_equal(outs[0][k], outs[1][k]) and np.array_equal(outs[0][k], outs[2][k]), k
