"""CPU checks of bench.py's host logic: the clock record keeps only samples
that arrived inside the timed region (or the first one after it started),
flags throttle reasons, the launch count follows the scan plan, and the
roofline byte counts are those the design states per token-head."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import chunked_gated_delta_gb300 as kda  # noqa: E402


def _line(mhz, reasons=("Not Active",) * 4):
    return "0, %d, 2070, 900.00 W, 0x0, %s" % (mhz, ", ".join(reasons))


def _sampler(samples, t0, t1):
    c = bench.ClockSampler(0)
    c.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0,
                            "kill": lambda self: None})()
    c.lines = samples
    c.t0, c.t1 = t0, t1
    return c


def test_clock_samples_inside_the_timed_region():
    samples = [(0.0, _line(1000)), (1.0, _line(2070)), (1.02, _line(2040)), (1.05, _line(2070)), (2.0, _line(500))]
    rec = _sampler(samples, 0.99, 1.04).stop()
    assert rec["window"] == "timed region" and rec["samples"] == 3
    assert rec["sm_mhz"] == 2070.0 and rec["sm_max_mhz"] == 2070.0 and rec["reasons"] == []


def test_short_region_takes_the_first_sample_after_its_start():
    samples = [(0.0, _line(800)), (0.5, _line(1900)), (0.8, _line(2070))]
    rec = _sampler(samples, 0.1, 0.12).stop()
    assert rec["window"].startswith("first sample") and rec["samples"] == 1 and rec["sm_mhz"] == 1900.0


def test_throttle_reasons_are_reported():
    hot = _line(1500, ("Active", "Not Active", "Not Active", "Active"))
    rec = _sampler([(1.0, hot)], 0.9, 1.1).stop()
    assert rec["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_launches_per_step_follow_the_plan():
    plain = kda.workspace_layout(kda.make_dims(4, 8192, 32, 128, 128))
    seg = kda.workspace_layout(kda.make_dims(1, 4096, 16, 128, 128))
    staged = kda.workspace_layout(kda.make_dims(1, 65536, 32, 128, 128))
    assert bench.launches_per_step(plain) == 3           # planner, intra, scan
    assert bench.launches_per_step(seg) == 5             # + map pass and combine
    assert bench.launches_per_step(staged) == 1 + 2 * 8  # planner + (intra, scan) per chunk range


def test_roofline_bytes_per_token_head():
    intra, scan = bench.bytes_per_token_head(128, 128)
    assert intra == 2 * 2 * 128 + 2 * 128 + 4 * 128 + 2 + 3 * 2 * 128 + 2 * 128 + 2 * 64 + 4 * 128 // 64  # 2442
    assert scan == 3 * 2 * 128 + 2 * 64 + 2 * 128 + 4 * 128 // 64 + 2 * 128                               # 1416
    assert intra + scan == 3858
    assert bench.flops_per_token_head(128, 128) == 180224


@pytest.mark.parametrize("dims", [(4, 8192, 32, 128, 128), (1, 65536, 32, 128, 128), (3, 1537, 32, 64, 128)])
def test_host_arena_of_time_slices(dims):
    """Fixed-length problems of 4096+ rows take the time-slice pipeline: the arena
    holds two slots of one slice (a fraction of the whole inputs) plus the
    workspace of the largest slice."""
    d = kda.make_dims(*dims)
    B, T, H, K, V = dims
    whole_io = B * T * H * (2 * K * 2 + V * 2 + K * 4 + 2 + V * 2)
    arena = kda.host_arena_size(d)
    assert 0 < arena < whole_io + kda.workspace_size(d)
    nt = (T + 63) // 64
    per = -(-nt // 8)
    slice_ws = kda.workspace_size(kda.make_dims(B, per * 64, H, K, V))
    assert arena >= slice_ws


def test_short_region_reports_the_clock_window():
    """A timed region shorter than the sampling period holds no sample; the
    clock-only window of untimed steps after it supplies the figure, labelled."""
    samples = [(0.0, _line(800)), (0.31, _line(2070)), (0.36, _line(2055)), (0.41, _line(2070)), (1.5, _line(900))]
    c = _sampler(samples, 0.10, 0.113)
    c.mark_window(0.3, 0.45)
    rec = c.stop()
    assert rec["samples_in_region"] == 0 and rec["samples_clock_window"] == 3
    assert rec["window"].startswith("clock window") and rec["samples"] == 3 and rec["sm_mhz"] == 2070.0


def test_percentiles_and_strict_roofline():
    assert bench.pct([4.0, 1.0, 3.0, 2.0], 0.5) == 2.5 and bench.pct([1.0], 0.9) == 1.0
    assert bench.pct(list(range(11)), 0.1) == 1.0 and bench.pct(list(range(11)), 0.9) == 9.0
    assert bench.strict_bytes_per_token_head(128, 128) == 1538
    r = bench.step_roofline(128, 128, 1000, 0, 1.0, 1000.0, 1000.0)
    assert r["bytes"] == 3858 * 1000 and r["strict_io_bytes"] == 1538 * 1000
    assert abs(r["frac_of_strict_io_bound"] - 1538e3 / 1e12 * 1e3) < 1e-12


def test_kernel_key_ignores_comments_only(tmp_path):
    """The key that ties a committed ncu traffic figure to a kernel source
    changes with the code and not with its comments or blank lines."""
    src = ('// header\n#include "h.cuh"\n/* block\n   comment */\n__global__ void k(int* p) {\n'
           '    const char* s = "a // b /* c */";  // trailing\n    char q = \'\\\'\';\n\n    p[0] = 1;\n}\n')
    headers = {n: "// only a comment\nint x_%d;\n" % i for i, n in enumerate(bench.KERNEL_HEADERS)}

    def key(text):
        d = tmp_path / str(abs(hash(text)))
        d.mkdir()
        for n, body in headers.items():
            (d / n).write_text(body)
        (d / "k.cu").write_text(text)
        return bench.source_sha(str(d / "k.cu"))

    base = key(src)
    assert key(src.replace("// trailing", "// another remark").replace("// header", "")) == base
    assert key(src.replace("\n\n", "\n\n\n")) == base
    assert key(src.replace("p[0] = 1;", "p[0] = 2;")) != base
    assert key(src.replace('"a // b /* c */"', '"a // b"')) != base  # literals are code
    assert "// b /* c */" in bench.code_text(src) and "trailing" not in bench.code_text(src)
