"""The committed DRAM-traffic captures (profiles/traffic.json) that bench.py
reports as `roofline.traffic`: well formed, scaled by the number of cells,
and taken on the kernel sources as they stand (a capture goes stale, and the
bench reports null, as soon as the code of a captured source changes)."""
import copy
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402

TRAFFIC = os.path.join(bench.ROOT, "profiles", "traffic.json")
HEADLINE_CELLS = 1024 * 1024 * 128


def load():
    with open(TRAFFIC) as f:
        return json.load(f)


def test_captures_are_well_formed_and_scaled():
    t = load()
    seen = set()
    for c in t["captures"]:
        key = (c["layout"], c["factors"], c["az_form"])
        assert key not in seen
        seen.add(key)
        assert c["full_cells"] % c["captured_cells"] == 0
        scale = c["full_cells"] // c["captured_cells"]
        for role in ("spmv_fused", "precond_fused"):
            k = c["kernels"][role]
            assert k["captured_read"] > 0 and k["captured_write"] > 0
            assert abs(k["bytes_per_launch"] - scale * (k["captured_read"] + k["captured_write"])) \
                <= scale
    assert ("tiled", "stored", "residual") in seen   # the bench's default configuration


def test_captures_match_the_current_sources():
    for c in load()["captures"]:
        assert c["sha256"] == bench.sources_sha256(c["sources"]), (c["layout"], c["az_form"])
    # the headline's dominant kernel has a traffic figure, about 79 bytes per cell
    b = bench.measured_traffic("spmv_fused", HEADLINE_CELLS, "tiled", "stored", "residual")
    assert b is not None and 70 < b / HEADLINE_CELLS < 90


def test_a_code_change_makes_the_capture_stale(tmp_path, monkeypatch):
    t = load()
    c = copy.deepcopy(t)
    c["captures"][0]["sha256"] = "0" * 64
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "traffic.json").write_text(json.dumps(c))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    cap = t["captures"][0]
    # sources_sha256 reads the kernel sources under ROOT: point it back at the repository's
    monkeypatch.setattr(bench, "sources_sha256", lambda names: cap["sha256"])
    assert bench.measured_traffic("spmv_fused", cap["full_cells"], cap["layout"], cap["factors"],
                                  cap["az_form"]) is None
    # a comment-only edit keeps the hash: comments and whitespace are removed before hashing
    monkeypatch.undo()
    src = os.path.join(bench.ROOT, "matrix_free_pcg_gb300", "csrc", cap["sources"][0])
    with open(src) as f:
        text = f.read()
    h0 = bench.sources_sha256(cap["sources"])
    pkg = tmp_path / "matrix_free_pcg_gb300" / "csrc"
    pkg.mkdir(parents=True)
    for name in cap["sources"]:
        with open(os.path.join(bench.ROOT, "matrix_free_pcg_gb300", "csrc", name)) as f:
            body = f.read()
        if name == cap["sources"][0]:
            body = "// a note\n" + body.replace("\n", "  \n", 3)
        (pkg / name).write_text(body)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.sources_sha256(cap["sources"]) == h0
    (pkg / cap["sources"][0]).write_text(text + "\nint an_extra_symbol;\n")
    assert bench.sources_sha256(cap["sources"]) != h0
