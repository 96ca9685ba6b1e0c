"""The step timeline's host side on CPU: medians of the trace tables per row,
rows a step did not stamp left out, and the printed busy column (kernels from
the later of their wait and the previous kernel's exit; points inside the
sampling kernel from the previous point, the first from the kernel's wait)."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

# (row, entry, wait done, exit) in us after the prologue's entry
KERNELS = [(0, 0.0, 0.0, 7.0), (1, 5.0, 9.0, 21.0), (2, 17.0, 22.0, 32.0), (3, 24.0, 33.0, 40.0),
           (4, 26.0, 41.0, 54.0), (5, 46.0, 55.0, 90.0), (6, 84.0, 91.0, 112.0), (7, 92.0, 114.0, 117.0),
           (8, 106.0, 118.0, 300.0), (10, 114.0, 301.0, 313.0), (11, 284.0, 312.5, 321.0)]
POINTS = [(25, 301.5, 302.0), (26, 305.0, 305.5), (27, 305.6, 306.0), (28, 307.0, 309.0),
          (29, 310.0, 310.0), (30, 312.0, 312.0)]


def _tables(steps=5, base=10 ** 9):
    rng = np.random.default_rng(0)
    a = np.zeros((steps, 32, 3), dtype=np.float64)
    a[:, :, 0:2] = 2 ** 62
    for s in range(steps):
        t0 = base + s * 10 ** 6
        jit = rng.integers(-200, 200)  # ns: the median takes the middle step
        for k, ent, wt, ex in KERNELS:
            a[s, k] = [t0 + ent * 1e3 + jit, t0 + wt * 1e3 + jit, t0 + ex * 1e3 + jit]
        a[s, 0, 0] = t0
        for k, first, last in POINTS:
            a[s, k] = [t0 + first * 1e3 + jit, t0 + first * 1e3 + jit, t0 + last * 1e3 + jit]
    return a


def test_rows_are_medians_in_timeline_order():
    a = _tables()
    out = bench.timeline_rows(a)
    rows = [k for k, *_ in out]
    assert rows == [k for k in bench.TIMELINE_ORDER if k in {r[0] for r in KERNELS} | {p[0] for p in POINTS}]
    assert 9 not in rows and 24 not in rows  # no acceptance kernel, no LM-head fixup in this step
    want = {k: (e, w, x) for k, e, w, x in KERNELS}
    want.update({k: (f, f, last) for k, f, last in POINTS})
    for k, ent, wt, ex in out:
        assert np.allclose((ent, wt, ex), want[k], atol=0.25), (k, ent, wt, ex)


def test_a_row_missing_in_one_step_is_left_out():
    a = _tables()
    a[2, 26, 2] = 0  # one step never reached the point
    assert 26 not in [k for k, *_ in bench.timeline_rows(a)]


def test_printed_busy_column(capsys):
    out = [(k, e, w, x) for k, e, w, x in KERNELS if k != 11] + \
          [(k, f, f, last) for k, f, last in POINTS] + [(11, 284.0, 312.5, 321.0)]
    out.sort(key=lambda r: bench.TIMELINE_ORDER.index(r[0]))
    bench.print_timeline("synthetic", 320.0, out)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("| ") and "---" not in ln]
    busy = {ln.split(" | ")[0][2:]: float(ln.rstrip(" |").split(" | ")[-1]) for ln in lines[1:]}
    assert busy["LM-head GEMM"] == 300.0 - 118.0
    assert busy["sampling"] == 313.0 - 301.0
    # the first point counts from the sampling kernel's wait, the others from the previous point
    assert busy["- sampling: status read"] == 302.0 - 301.0
    assert busy["- sampling: row statistics merged"] == 305.5 - 302.0
    assert busy["- sampling: draw's chunk found"] == 312.0 - 310.0
    # the kernel after the points counts from the sampling kernel's exit (313.0,
    # after its own wait stamp here), not from the last point (312.0)
    assert busy["realignment"] == 321.0 - 313.0
    assert "| - sampling: status read | 301.5 | - | 302.0 |" in "\n".join(lines)


def test_a_kernel_whose_blocks_all_left_before_the_wait():
    """A fixup kernel with no cut tile: every block leaves before its wait, so
    the wait stamp keeps its initial value; the row shows no wait and adds
    nothing to the step, and the next kernel still counts from the GEMM."""
    a = _tables()
    for s in range(a.shape[0]):
        t0 = a[s, 0, 0]
        a[s, 17] = [t0 + 6.0e3, 2 ** 62, t0 + 8.0e3]  # the QKV GEMM's fixup: entry and exit only
    out = bench.timeline_rows(a)
    row = [r for r in out if r[0] == 17]
    assert len(row) == 1 and row[0][2] is None
    import io
    import contextlib
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.print_timeline("synthetic", 320.0, out)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("| ") and "---" not in ln]
    busy = {ln.split(" | ")[0][2:]: float(ln.rstrip(" |").split(" | ")[-1]) for ln in lines[1:]}
    assert busy["QKV GEMM fixup"] == 0.0
    assert busy["attention"] == 32.0 - 22.0
    assert "| QKV GEMM fixup | 6.0 | - | 8.0 |" in "\n".join(lines)
