"""bench.py reports roofline.traffic from profiles/traffic.json only while the kernel sources it
was measured on are unchanged (their sha256 recorded beside the counters)."""
import hashlib
import json
import os
import shutil

import bench


def _tree(tmp_path, sources, edit=None):
    for src in sources:
        dst = tmp_path / src
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, src), dst)
    if edit:
        with open(tmp_path / edit, "a") as fh:
            fh.write("\n// changed\n")
    return tmp_path


def test_traffic_needs_the_measured_sources(tmp_path, monkeypatch):
    srcs = ["moe_speculative_decoding_gb300/csrc/expert_tc.cu", "moe_speculative_decoding_gb300/csrc/common.cuh"]
    h = hashlib.sha256()
    for s in srcs:
        with open(os.path.join(bench.ROOT, s), "rb") as fh:
            h.update(fh.read())
    entry = {"sources": srcs, "sources_sha256": h.hexdigest(), "dram_bytes_per_launch": 123}
    for edit, expect in ((None, 123), (srcs[0], None)):
        root = tmp_path / ("edited" if edit else "same")
        _tree(root, srcs, edit)
        (root / "profiles").mkdir()
        (root / "profiles" / "traffic.json").write_text(json.dumps({"k": entry}))
        monkeypatch.setattr(bench, "ROOT", str(root))
        got = bench.kernel_traffic("k")
        assert (got["dram_bytes_per_launch"] if got else None) == expect
        assert bench.kernel_traffic("other") is None   # no entry for that kernel


def test_no_profile_no_traffic(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("expert_tc_kernel") is None
