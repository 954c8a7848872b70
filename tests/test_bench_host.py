"""bench.py's host logic, no GPU: the clock record keeps only the nvidia-smi
samples taken inside the timed region; the profile digest ignores comments but
not code; the byte model gives the documented per-launch figures."""
import datetime
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def _line(t, sm, mx=2070, reasons=("Not Active",) * 4):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([ts, "0", str(sm), str(mx), "900.00", "0x0000000000000000", *reasons])


def test_samples_inside_the_region_only():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.10, 1000), _line(t0 + 0.05, 2070), _line(t0 + 0.10, 2040),
             _line(t0 + 0.15, 2070), _line(t0 + 0.40, 900, reasons=("Active",) + ("Not Active",) * 3)]
    r = bench.Clocks.summarize(lines, t0, t0 + 0.2)
    assert r["samples"] == 3
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == []  # the hw_slowdown sample lies after the region


def test_reasons_inside_the_region_are_reported():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.05, 1980, reasons=("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 0.10, 1900, reasons=("Not Active", "Active", "Not Active", "Not Active"))]
    r = bench.Clocks.summarize(lines, t0, t0 + 0.2)
    assert r["samples"] == 2
    assert r["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_short_region_falls_back_to_the_nearest_sample():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 1.0, 1500), _line(t0 + 0.06, 2055), _line(t0 + 1.0, 1400)]
    r = bench.Clocks.summarize(lines, t0, t0 + 0.01)
    assert r["samples"] == 0 and r["sm_mhz"] == 2055.0


def test_unparsable_output_gives_no_record():
    assert bench.Clocks.summarize(["No devices were found"], 0.0, 1.0) is None
    assert bench.Clocks.summarize([], 0.0, 1.0) is None


def test_source_digest_ignores_comments_not_code(tmp_path):
    base = 'int f(int x) {  // the CTA\'s "row"\n    /* block\n comment */ return x + 1;\n}\nconst char *s = "a // b";\n'
    p = tmp_path / "k.cu"
    p.write_text(base)
    d0 = bench.source_digest(str(p))
    p.write_text(base.replace("the CTA's", "every CTA's").replace("block\n", "other\n\n"))
    assert bench.source_digest(str(p)) == d0  # comments and blank lines only
    p.write_text(base.replace("x + 1", "x + 2"))
    assert bench.source_digest(str(p)) != d0  # code
    p.write_text(base.replace('"a // b"', '"a // c"'))
    assert bench.source_digest(str(p)) != d0  # "//" inside a string is code


def test_byte_model_matches_the_documented_figures():
    """The roofline's algorithmic bytes per launch for the FlyGPT shape are the
    ones the design notes quote (9.42 GB forward, 10.04 GB backward); the
    gathered rows (4EB per microstep) are most of them."""
    fwd, bwd = bench.byte_model(5000, 524324, 32, 64, 2, 64)
    assert (fwd, bwd) == (9_417_761_280, 10_035_540_480)
    gathered = 64 * 2 * 4 * 524324 * 32
    assert 0.9 < gathered / fwd < 1.0 and 0.85 < gathered / bwd < 1.0


def test_step_roofline_takes_the_slower_bound():
    # FlyGPT-like: 19.45 GB at L2 over 18,000 GB/s beats 0.43 GB over 6,673 GB/s
    r = bench.step_roofline(19.45e9, 0.43e9, 18000.0, 6673.5, 2.4)
    assert r["bound"] == "l2" and abs(r["roofline_ms"] - 19.45 / 18.0) < 1e-9
    assert abs(r["frac"] - (19.45 / 18.0) / 2.4) < 1e-9
    r = bench.step_roofline(1e9, 30e9, 18000.0, 6000.0, 10.0)
    assert r["bound"] == "hbm" and abs(r["roofline_ms"] - 5.0) < 1e-9 and abs(r["frac"] - 0.5) < 1e-9


def test_memory_figures_add_up():
    import bench
    m = bench.memory_figures(N=10, E=30, B=4, T=3, n_in=2, graph_bytes=1000, saved_b=500,
                             scratch_b=200, ckpt_b=100, scratch_rc_b=300)
    io = 4 * ((30 + 20 + 24 + 40) + 2 * 120 + (30 + 20 + 24 + 40))
    assert m["io_bytes"] == io
    assert m["step_bytes"] == 1000 + io + 500 + 200
    assert m["recompute"]["step_bytes"] == 1000 + io + 100 + 300


def test_l2_sweep_shapes_are_accepted_by_the_probe():
    """Every swept shape satisfies ck_probe_read_shape's documented limits, so
    the bench's sweep cannot be cut short by a refused shape."""
    import bench
    for lb, depth, thr, cps in bench.L2_SWEEP:
        assert lb in (16, 32) and depth in (2, 4, 8, 16) and thr in (128, 256, 512, 1024)
        assert 1 <= cps and thr * cps <= 2048
        assert not (depth == 16 and thr > 512)
    assert any(lb == 32 for lb, *_ in bench.L2_SWEEP)
    # one pass of a 160-SM grid stays within half the buffer
    for lb, depth, thr, cps in bench.L2_SWEEP:
        assert lb * depth * thr * cps * 160 <= bench.L2_SWEEP_BYTES // 2
