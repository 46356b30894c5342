"""Host-side logic of bench.py that needs no GPU: the DRAM-traffic figure of the
roofline line comes from the committed ncu capture, scaled by the groups one
group-kernel launch chains, and is withheld when the kernel source or the
shape differs from the captured one."""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traffic_scales_with_the_groups_of_a_launch():
    b = _bench()
    with open(b.TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    shape = rec["captured_shape"]
    per = rec["dram_bytes_per_group"]
    if rec["kernel_sha256_16"] != b.kernel_hash():
        pytest.skip("the group kernel changed since the committed ncu capture: the bench reports "
                    "traffic null until profiles/group_kernel_traffic.json is refreshed")
    assert per * rec["captured_groups"] <= rec["dram_bytes_captured"] < (per + 1) * rec["captured_groups"]
    for groups in (1, 4, 16):
        assert b.stored_traffic(groups, rec["captured_chunk"], shape["d"], shape["f"]) == per * groups


def test_traffic_withheld_for_another_shape_or_kernel(tmp_path, monkeypatch):
    b = _bench()
    with open(b.TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    shape = rec["captured_shape"]
    assert b.stored_traffic(16, rec["captured_chunk"] // 2, shape["d"], shape["f"]) is None
    assert b.stored_traffic(16, rec["captured_chunk"], shape["d"] * 2, shape["f"]) is None
    stale = dict(rec, kernel_sha256_16="0" * 16)
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(stale))
    monkeypatch.setattr(b, "TRAFFIC_FILE", str(path))
    assert b.stored_traffic(16, rec["captured_chunk"], shape["d"], shape["f"]) is None
