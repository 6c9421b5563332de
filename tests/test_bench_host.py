"""bench.py host logic that needs no GPU: the staleness check of the stored
level-0 DRAM counters."""
import json
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402

CSRC = os.path.join(ROOT, "elliptic_curve_scalar_gb300", "csrc")


def _local_includes(name, seen):
    if name in seen:
        return
    seen.add(name)
    with open(os.path.join(CSRC, name)) as f:
        for inc in re.findall(r'^\s*#include\s+"([^"]+)"', f.read(), re.M):
            _local_includes(inc, seen)


def test_digest_covers_every_header_of_the_kernel():
    seen = set()
    _local_includes("msm_accum.cu", seen)
    assert seen == set(bench.LEVEL0_SOURCES)


def test_digest_follows_every_source():
    base = {name: b"x" for name in bench.LEVEL0_SOURCES}
    d0 = bench.level0_sources_digest(lambda name: base[name])
    assert d0 == bench.level0_sources_digest(lambda name: base[name])
    for name in bench.LEVEL0_SOURCES:
        changed = dict(base, **{name: b"y"})
        assert bench.level0_sources_digest(lambda nm: changed[nm]) != d0


def test_traffic_only_for_the_build_it_was_taken_on(tmp_path):
    prof = tmp_path / "traffic.json"
    prof.write_text(json.dumps({"n2p16_Sauto": 123, "sources_sha256": bench.level0_sources_digest()}))
    assert bench.level0_traffic("n2p16_Sauto", str(prof)) == (123, None)
    assert bench.level0_traffic("n2p20_Sauto", str(prof)) == (None, None)
    prof.write_text(json.dumps({"n2p16_Sauto": 123, "sources_sha256": "0" * 64}))
    assert bench.level0_traffic("n2p16_Sauto", str(prof)) == (None, 123)
    assert bench.level0_traffic("n2p16_Sauto", str(tmp_path / "missing.json")) == (None, None)


def _row(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return "0, %s, %s, 612.40, 0x0000000000000000, %s, %s, %s, %s\n" % (sm, mx, hw, hwt, swt, cap)


def test_clock_summary_of_a_clean_run():
    c = bench.summarize_clocks([_row(2070, 2070), _row(2055, 2070), _row(2070, 2070)])
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}


def test_clock_summary_reports_every_active_reason():
    lines = [_row(1980, 2070, cap="Active"), _row(1500, 2070, hwt="Active"), _row(2070, 2070),
             "garbled line\n", _row("[N/A]", 2070)]
    c = bench.summarize_clocks(lines)
    assert c["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert c["samples"] == 4 and c["sm_mhz"] == 1980.0 and c["sm_max_mhz"] == 2070.0


def test_clock_summary_without_samples():
    assert bench.summarize_clocks([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_clock_sampler_without_nvidia_smi_reports_no_samples(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", "")
    s = bench.ClockSampler(tmpdir=str(tmp_path))
    c = s.stop()
    assert c["samples"] == 0 and c["reasons"] == []
    assert not list(tmp_path.iterdir())  # the sample file is removed
