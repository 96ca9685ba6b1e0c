import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # keep GPU tests from running (and failing) on a machine without a GPU
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def nine_b_weights():
    """The 9B-class layer + LM head (seed 2) on the host and on cuda:0, shared by the GPU modules."""
    import torch
    assert torch.cuda.is_available()
    import workloads as wl
    from workloads import device as wd
    W = wl.make_weights(wl.NINE_B, 2)
    return W, wd.weights_to_device(W)


@pytest.fixture(scope="session")
def nine_b_int4():
    """The 9B-class layer with int4 group-32 projections (seed 5), bf16 LM head, host and cuda:0."""
    import torch
    assert torch.cuda.is_available()
    import workloads as wl
    from workloads import device as wd
    W = wl.make_weights(wl.NINE_B, 5, fmt="int4")
    return W, wd.weights_to_device(W)


def pytest_terminal_summary(terminalreporter):
    """How often the GPU step comparisons explained a row by another bf16
    rounding at a tie (tiny model only; the 9B-class checks never do)."""
    mod = sys.modules.get("tests.gpu_helpers")
    if mod is None:
        return
    used = getattr(mod, "FLIPS_USED", [])
    nine_b = sum(1 for h, _, _ in used if h > 256)
    terminalreporter.write_line(f"parity: other roundings used {len(used)} (tiny model {len(used) - nine_b}, "
                                f"9B-class layer {nine_b})")
