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
