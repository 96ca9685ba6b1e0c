"""The C-ABI library loads, exports every function include/sdv.h declares, and
the Python binding's ctypes structs have the header's layout (CPU only).
"""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdv.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verify_ragged_gb300 import _abi
    if not os.path.exists(_abi.LIB_PATH):
        from speculative_decoding_verify_ragged_gb300 import build
        build.build()
    return _abi.load_library()


HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


def test_library_exports_every_declared_symbol(lib):
    from speculative_decoding_verify_ragged_gb300 import _abi
    names = sorted({n for h in HEADERS for n in _abi.header_symbols(h)})
    assert len(names) >= 20 and "sdv_admit" in names and "sdv_sched_plan" in names
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


PROBE = r"""
#include <stdio.h>
#include <stddef.h>
#include "sdv_sched.h"
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("sdv_config %zu\nsdv_weights %zu\nsdv_batch %zu\nsdv_result %zu\n",
         sizeof(sdv_config), sizeof(sdv_weights), sizeof(sdv_batch), sizeof(sdv_result));
  printf("sdv_admission %zu\nsdv_sched_config %zu\nsdv_sched_step %zu\nsdv_sched_stats %zu\n",
         sizeof(sdv_admission), sizeof(sdv_sched_config), sizeof(sdv_sched_step), sizeof(sdv_sched_stats));
  F(sdv_admission, max_pages_per_seq) F(sdv_admission, num_free) F(sdv_sched_stats, live)
  F(sdv_config, rope_theta) F(sdv_weights, g_final) F(sdv_batch, num_pool_pages)
  F(sdv_batch, max_pages_per_seq) F(sdv_batch, gen_limits) F(sdv_batch, tree_parents) F(sdv_result, logits) F(sdv_result, status)
  return 0;
}
"""


def test_ctypes_layout_matches_header(tmp_path):
    from speculative_decoding_verify_ragged_gb300 import _abi
    src = tmp_path / "probe.c"
    src.write_text(PROBE)
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    vals = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                          check=True).stdout.splitlines())
    assert int(vals["sdv_config"]) == ctypes.sizeof(_abi.SdvConfig)
    assert int(vals["sdv_weights"]) == ctypes.sizeof(_abi.SdvWeights)
    assert int(vals["sdv_batch"]) == ctypes.sizeof(_abi.SdvBatch)
    assert int(vals["sdv_result"]) == ctypes.sizeof(_abi.SdvResult)
    assert int(vals["sdv_config.rope_theta"]) == _abi.SdvConfig.rope_theta.offset
    assert int(vals["sdv_weights.g_final"]) == _abi.SdvWeights.g_final.offset
    assert int(vals["sdv_batch.num_pool_pages"]) == _abi.SdvBatch.num_pool_pages.offset
    assert int(vals["sdv_batch.max_pages_per_seq"]) == _abi.SdvBatch.max_pages_per_seq.offset
    assert int(vals["sdv_batch.gen_limits"]) == _abi.SdvBatch.gen_limits.offset
    assert int(vals["sdv_batch.tree_parents"]) == _abi.SdvBatch.tree_parents.offset
    assert int(vals["sdv_result.logits"]) == _abi.SdvResult.logits.offset
    assert int(vals["sdv_result.status"]) == _abi.SdvResult.status.offset
    assert int(vals["sdv_admission"]) == ctypes.sizeof(_abi.SdvAdmission)
    assert int(vals["sdv_sched_config"]) == ctypes.sizeof(_abi.SdvSchedConfig)
    assert int(vals["sdv_sched_step"]) == ctypes.sizeof(_abi.SdvSchedStep)
    assert int(vals["sdv_sched_stats"]) == ctypes.sizeof(_abi.SdvSchedStats)
    assert int(vals["sdv_admission.max_pages_per_seq"]) == _abi.SdvAdmission.max_pages_per_seq.offset
    assert int(vals["sdv_admission.num_free"]) == _abi.SdvAdmission.num_free.offset
    assert int(vals["sdv_sched_stats.live"]) == _abi.SdvSchedStats.live.offset


def test_host_errors_without_device(lib):
    """Null and malformed arguments are refused before any CUDA call."""
    from speculative_decoding_verify_ragged_gb300 import _abi
    h = ctypes.c_void_p()
    assert lib.sdv_create(None, None, None, 0, 1, 1, ctypes.byref(h)) == _abi.SDV_ERR_INVALID_ARG
    cfg = _abi.SdvConfig(256, 4, 2, 96, 768, 1024, 16, 3, 0, 1e-6, 1e6)   # head_dim 96: no kernel
    w = _abi.SdvWeights()
    assert lib.sdv_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.c_void_p(256), 1 << 20, 8, 2,
                          ctypes.byref(h)) == _abi.SDV_ERR_UNSUPPORTED
    assert lib.sdv_verify_step(None, None, None, None) == _abi.SDV_ERR_INVALID_ARG
    assert lib.sdv_accept(None, None, None, None, None) == _abi.SDV_ERR_INVALID_ARG
    assert lib.sdv_realign(None, None, None, None) == _abi.SDV_ERR_INVALID_ARG
    assert lib.sdv_linear(None, 0, None, 0, None, 1, None) == _abi.SDV_ERR_INVALID_ARG
    assert lib.sdv_attention(None, None, None, None, None, None) == _abi.SDV_ERR_INVALID_ARG
    assert lib.sdv_read_status(None, None, None) == _abi.SDV_ERR_INVALID_ARG
    assert lib.sdv_set_gemm_path(None, 0) == _abi.SDV_ERR_INVALID_ARG
    assert lib.sdv_admit(None, None, None, None) == _abi.SDV_ERR_INVALID_ARG
    bad = _abi.SdvConfig(256, 4, 3, 64, 768, 1024, 16, 3, 0, 1e-6, 1e6)     # n_q not a multiple of n_kv
    assert lib.sdv_workspace_size(ctypes.byref(bad), 8, 2) == 0
    # a vocabulary past the sampling chunk table (2048 chunks of 512 entries)
    big = _abi.SdvConfig(256, 4, 2, 64, 768, 2048 * 512 + 1, 16, 3, 0, 1e-6, 1e6)
    assert lib.sdv_workspace_size(ctypes.byref(big), 8, 2) == 0


def test_product_has_no_cpu_fallback():
    """The binding raises when the library is missing; it never imports the oracle."""
    code = (
        "import sys, speculative_decoding_verify_ragged_gb300._abi as a\n"
        "try:\n"
        "    a.load_library('/nonexistent/libsdv.so')\n"
        "    sys.exit(1)\n"
        "except RuntimeError:\n"
        "    pass\n"
        "assert 'oracle' not in sys.modules and not any(m.startswith('oracle.') for m in sys.modules)\n"
    )
    subprocess.run([sys.executable, "-c", code], check=True, cwd=ROOT)
    pkg = os.path.join(ROOT, "speculative_decoding_verify_ragged_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_timeline_needs_the_trace_build():
    """The product library has no timeline stamps: sdv_trace_enable refuses
    (without touching the GPU)."""
    from speculative_decoding_verify_ragged_gb300 import _abi
    lib = _abi.load_library()
    assert lib.sdv_trace_enable(None) == _abi.SDV_ERR_UNSUPPORTED
