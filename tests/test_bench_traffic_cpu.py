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


def test_union_roofline_follows_the_kernels_path():
    """The union cost's bytes delivered per call: one word per node triple and the root with the
    table (18 nodes, 48 layers, 2 words: 7 x 96 x 8 B per subset), one per node otherwise."""
    r = bench.union_roofline(18, 48, 2, 1 << 18, 46.6e-6, 152)
    assert r["path"] == "node-triple table" and r["delivered_bytes_per_call"] == (1 << 18) * 7 * 96 * 8
    assert abs(r["peak_tbps"] - 152 * 128 * 2.07e9 / 1e12) < 0.01 and 0 < r["frac"] < 1
    odd = bench.union_roofline(10, 27, 1, 1024, 1e-5, 152)      # L*W odd
    big = bench.union_roofline(12, 400, 2, 800, 1e-5, 152)      # table beside the root above 200 KB
    assert odd["path"] == big["path"] == "broadcast node loop"
    assert odd["delivered_bytes_per_call"] == 1024 * 11 * 27 * 8
