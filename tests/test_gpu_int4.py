"""The layer with int4 group-32 weights (fp16 scales) against the oracle.

The oracle dequantises exactly (w = s * q in float64); the kernel multiplies
the exact codes in bf16 and applies each group's scale to the group's fp32
partial sum, so the linear results carry only fp32 summation error.  Full
steps check the same logits / probabilities / decisions bar as the bf16
layer (the LM head stays bf16).
"""
import numpy as np
import pytest

from oracle import verify_step as o
import workloads as wl
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

NAMES = ["qkv", "o", "gate", "up", "down"]


@pytest.fixture(scope="module")
def tiny_int4():
    import torch
    assert torch.cuda.is_available()
    from workloads import device as wd
    W = wl.make_weights(wl.TINY, 5, fmt="int4")
    Wd = wd.weights_to_device(W)
    eng = gh.engine_for(wl.TINY, 3, Wd, max_rows=160, max_slots=40, fmt="int4")
    return W, Wd, eng


@pytest.mark.parametrize("xfmt", ["bf16", "f32"])
@pytest.mark.parametrize("rows", [1, 5, 8, 9, 16, 17, 32, 33, 64, 100, 160])
@pytest.mark.parametrize("which", [0, 1, 2, 3, 4])
def test_linear_int4(tiny_int4, rows, which, xfmt):
    import torch
    W, _, eng = tiny_int4
    w = W.proj[NAMES[which]]
    wf = o.dequant_int4_g32(*w)
    K = wf.shape[1]
    x32 = np.random.default_rng(2000 + rows * 10 + which).standard_normal((rows, K)).astype(np.float32)
    if xfmt == "bf16":
        x = wl.f32_to_bf16_bits(x32)
        xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
        xf = o.bf16_to_f64(x)
    else:
        xd = torch.from_numpy(x32).cuda()
        xf = x32.astype(np.float64)
    y = torch.empty((rows, wf.shape[0]), dtype=torch.float32, device="cuda")
    eng.linear(which, xd, y)
    torch.cuda.synchronize()
    ref = o.linear(xf, w)
    scale = np.sqrt((xf ** 2).sum(1)).max() * np.abs(wf).max()
    tol = 1e-5 if xfmt == "bf16" else 3e-5
    assert np.abs(y.cpu().numpy() - ref).max() <= tol * scale + 1e-6


def test_linear_int4_sign_and_nibble_order(tiny_int4):
    """Hand-made codes: every code value in both nibbles, scales of both signs."""
    import torch
    from workloads import device as wd
    W, _, _ = tiny_int4
    dims = wl.TINY
    codes = (np.arange(dims["hidden"]) % 16 - 8).astype(np.int8)          # -8..7 repeating along k
    n_qkv = (dims["n_q"] + 2 * dims["n_kv"]) * dims["head_dim"]
    q = np.tile(codes, (n_qkv, 1))
    q[1::2] = q[1::2, ::-1]                                                 # odd rows: reversed order
    u = (q.astype(np.int16) & 0xF).astype(np.uint8)
    packed = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    s = np.where(np.arange(n_qkv)[:, None] % 3 == 0, -0.5, 0.25) * (1 + np.arange(dims["hidden"] // 32))[None, :]
    scales = s.astype(np.float16).view(np.uint16)
    W2 = wl.Weights(dims=W.dims, fmt="int4", emb=W.emb, g_attn=W.g_attn, g_ffn=W.g_ffn, g_final=W.g_final,
                    w_lm=W.w_lm, proj=dict(W.proj, qkv=(packed, scales)))
    eng = gh.engine_for(wl.TINY, 3, wd.weights_to_device(W2), max_rows=16, max_slots=4, fmt="int4")
    x = np.eye(dims["hidden"], dtype=np.float32)[:16] + 0.001 * np.arange(16, dtype=np.float32)[:, None]
    y = torch.empty((16, n_qkv), dtype=torch.float32, device="cuda")
    eng.linear(0, torch.from_numpy(x).cuda(), y)
    torch.cuda.synchronize()
    ref = o.linear(x.astype(np.float64), (packed, scales))
    assert np.abs(y.cpu().numpy() - ref).max() <= 1e-5 * np.abs(ref).max()


def test_step_tiny_int4(tiny_int4):
    from tests.test_gpu_parity import _full_step_check
    W, _, eng = tiny_int4
    b1 = wl.make_batch(wl.TINY, 51, seq_lens=[128, 128], draft_lens=[3, 1], gamma_max=3, extra_pages=4)
    _full_step_check(eng, W, b1, "tiny-int4")
    lens = [0, 37, 128, 5, 200, 64, 91, 16]
    gam = [3, 0, 2, 1, 3, 3, 2, 0]
    b2 = wl.make_batch(wl.TINY, 52, seq_lens=lens, draft_lens=gam, gamma_max=3, extra_pages=10)
    _full_step_check(eng, W, b2, "tiny-int4-ragged")
    lens = list(range(3, 400, 11))[:36]
    gam = [(5 * i) % 4 for i in range(36)]
    b3 = wl.make_batch(wl.TINY, 53, seq_lens=lens, draft_lens=gam, gamma_max=3, extra_pages=40)
    assert b3.R > 64
    _full_step_check(eng, W, b3, "tiny-int4-wide")


def test_step_nine_b_int4(nine_b_int4):
    """9B-class int4 layer: a swarm-like ragged batch (contexts 1k..16k, gamma 0..3)."""
    from tests.test_gpu_parity import _retargeted
    from tests.test_gpu_parity import _full_step_check
    W, Wd = nine_b_int4
    eng = gh.engine_for(wl.NINE_B, 3, Wd, max_rows=64, max_slots=16, fmt="int4")
    g = np.random.default_rng(55)
    lens = g.integers(1024, 16385, size=6)
    gam = [3, 0, 2, 1, 3, 2]
    batch = wl.make_batch(wl.NINE_B, 5, seq_lens=lens, draft_lens=gam, gamma_max=3,
                          alphas=[0.97, 0.8, 0.14, 0.8, 0.97, 0.14], extra_pages=12)
    _full_step_check(eng, W, _retargeted(batch, W, 5), "nine-b-int4")


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("rows", [16, 40, 128, 300])
@pytest.mark.parametrize("which", [0, 2, 4])
def test_linear_int4_nine_b_both_kernels(nine_b_int4, rows, which, path):
    """9B-class int4 projections through the mma.sync (path 1) and tcgen05 (path 2)
    kernels, fp32 activations, on sampled output columns (all rows)."""
    import torch
    W, Wd = nine_b_int4
    eng = gh.engine_for(wl.NINE_B, 3, Wd, max_rows=320, max_slots=16, fmt="int4")
    eng.set_gemm_path(path)
    w = W.proj[NAMES[which]]
    N, K = w[0].shape[0], w[0].shape[1] * 2
    x32 = np.random.default_rng(7000 + rows + which).standard_normal((rows, K)).astype(np.float32)
    y = torch.empty((rows, N), dtype=torch.float32, device="cuda")
    eng.linear(which, torch.from_numpy(x32).cuda(), y)
    torch.cuda.synchronize()
    cols = np.random.default_rng(rows * 7 + which).choice(N, size=48, replace=False)
    wf = o.dequant_int4_g32(w[0][cols], w[1][cols])
    ref = x32.astype(np.float64) @ wf.T
    got = y.cpu().numpy()[:, cols]
    scale = np.sqrt((x32.astype(np.float64) ** 2).sum(1)).max() * np.abs(wf).max()
    assert np.abs(got - ref).max() <= 3e-5 * scale
