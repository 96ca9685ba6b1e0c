"""The weight-streaming GEMM on the 5th-generation tensor cores (tcgen05, TMEM
accumulators) against the oracle, and against the mma.sync kernel.

Every GEMM of the step can run on either kernel (sdv_set_gemm_path); these
tests force each in turn, over activation tiles of 16..256 rows, ragged tails,
tiles split between CTAs (stream-K) and tiles kept whole, every fused epilogue
(fp32, residual, SwiGLU planes, QKV + RoPE + paged K/V scatter, LM head with
softmax statistics) and both activation formats (bf16, fp32 as two planes).
"""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

MMA_SYNC, TCGEN05 = 1, 2
NAMES = ["qkv", "o", "gate", "up", "down", None]


@pytest.fixture(scope="module")
def tiny_wide():
    import torch
    assert torch.cuda.is_available()
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 1)
    Wd = wd.weights_to_device(W)
    eng = gh.engine_for(wl.TINY, 3, Wd, max_rows=320, max_slots=80)
    return W, Wd, eng


def _linear(eng, which, x, fmt, path, N):
    import torch
    eng.set_gemm_path(path)
    try:
        if fmt == "bf16":
            xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
        else:
            xd = torch.from_numpy(x).cuda()
        y = torch.empty((x.shape[0], N), dtype=torch.float32, device="cuda")
        eng.linear(which, xd, y)
        torch.cuda.synchronize()
        return y.cpu().numpy()
    finally:
        eng.set_gemm_path(0)


@pytest.mark.parametrize("xfmt", ["bf16", "f32"])
@pytest.mark.parametrize("rows", [1, 16, 17, 33, 64, 65, 128, 160, 257, 320])
@pytest.mark.parametrize("which", [0, 1, 2, 3, 4, 5])
def test_linear_tcgen05(tiny_wide, rows, which, xfmt):
    W, _, eng = tiny_wide
    w = W.proj[NAMES[which]] if NAMES[which] else W.w_lm
    K = w.shape[1]
    x32 = np.random.default_rng(1000 + rows * 10 + which).standard_normal((rows, K)).astype(np.float32)
    if xfmt == "bf16":
        x = wl.f32_to_bf16_bits(x32)
        xf = o.bf16_to_f64(x)
    else:
        x, xf = x32, x32.astype(np.float64)
    y = _linear(eng, which, x, xfmt, TCGEN05, w.shape[0])
    ref = o.linear(xf, w)
    # fp32 accumulation of K exact bf16 products; an fp32 operand enters as bf16 hi + lo
    scale = np.sqrt((xf ** 2).sum(1)).max() * np.abs(o.bf16_to_f64(w)).max()
    tol = 1e-5 if xfmt == "bf16" else 3e-5
    assert np.abs(y - ref).max() <= tol * scale + 1e-6
    # the two kernels differ only in the order of the fp32 sums
    y1 = _linear(eng, which, x, xfmt, MMA_SYNC, w.shape[0])
    assert np.abs(y - y1).max() <= 2 * tol * scale + 1e-6


@pytest.mark.parametrize("rows", [16, 24, 64, 100, 200])
def test_lm_head_full_size_tcgen05(nine_b_weights, rows):
    """151936 x 4096 LM head on the tensor cores: sampled columns against float64 dots."""
    W, Wd = nine_b_weights
    eng = gh.engine_for(wl.NINE_B, 7, Wd, max_rows=256, max_slots=8)
    g = np.random.default_rng(50 + rows)
    x = wl.f32_to_bf16_bits(g.standard_normal((rows, 4096)).astype(np.float32))
    y = _linear(eng, 5, x, "bf16", TCGEN05, wl.NINE_B["vocab"])
    cols = np.sort(g.choice(wl.NINE_B["vocab"], size=3000, replace=False))
    cols = np.concatenate([cols, [0, 127, 128, wl.NINE_B["vocab"] - 1]])
    ref = o.bf16_to_f64(x) @ o.bf16_to_f64(W.w_lm[cols]).T
    assert np.abs(y[:, cols] - ref).max() <= 2e-5 * np.abs(ref).max()


def _step_both_paths(eng, W, batch, name):
    """Full step with the GEMMs forced onto tcgen05: oracle parity, and agreement with mma.sync."""
    from tests.test_gpu_parity import _full_step_check
    eng.set_gemm_path(TCGEN05)
    try:
        _full_step_check(eng, W, batch, name)
    finally:
        eng.set_gemm_path(0)


def test_step_tiny_tcgen05(tiny_wide):
    W, _, eng = tiny_wide
    _step_both_paths(eng, W, wl.workload1(), "tiny-tc")
    lens = list(range(0, 400, 7))[:57]
    gam = [(3 * i) % 4 for i in range(57)]
    batch = wl.make_batch(wl.TINY, 31, seq_lens=lens, draft_lens=gam, gamma_max=3, extra_pages=80)
    assert batch.R > 128
    _step_both_paths(eng, W, batch, "tiny-wide-tc")


def test_step_eight_agents_tcgen05(nine_b_weights):
    from tests.test_gpu_parity import _retargeted
    W, Wd = nine_b_weights
    eng = gh.engine_for(wl.NINE_B, 7, Wd, max_rows=64, max_slots=16)
    lens, gam, alphas = wl.workload3_shape()
    batch = wl.make_batch(wl.NINE_B, 3, seq_lens=lens, draft_lens=gam, gamma_max=7, alphas=alphas,
                          extra_pages=16)
    _step_both_paths(eng, W, _retargeted(batch, W, 3), "workload3-tc")


def test_gemm_path_argument(tiny_wide):
    from speculative_decoding_verify_ragged_gb300 import _abi
    _, _, eng = tiny_wide
    assert eng.lib.sdv_set_gemm_path(eng.handle, 3) == _abi.SDV_ERR_INVALID_ARG
    assert eng.lib.sdv_set_gemm_path(eng.handle, -1) == _abi.SDV_ERR_INVALID_ARG
    assert eng.lib.sdv_set_gemm_path(None, 0) == _abi.SDV_ERR_INVALID_ARG
