"""The DRAM-traffic record that bench.py's roofline object carries comes from a committed ncu
summary and is used only while the GEMM's code is the profiled code: the summary's source hash
must match the current source, and the hash ignores comments, so that re-wording a comment
keeps the record while any change to the code drops it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_record_is_for_the_current_gemm_code():
    with open(os.path.join(ROOT, "profiles", "qgemm_q4k_gateup_L148.json")) as f:
        rec = json.load(f)
    assert rec["gemm_src_sha1"] == bench.gemm_source_sha1(), "re-capture profiles/qgemm_q4k_gateup_L148.*"
    assert bench._traffic_for("qgemm_q4k_gateup_L148.json") == rec["dram_bytes_read"] + rec["dram_bytes_write"]


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "quantized_gemm_q8_gb300" / "csrc"
    csrc.mkdir(parents=True)
    base = {"qgemm.cuh": "// header\nint f(int x) {\n  return x + 1;  // add\n}\n",
            "ptx.cuh": "/* block\n comment */\n#pragma once\n"}

    def digest(files):
        for name, text in files.items():
            (csrc / name).write_text(text)
        monkeypatch.setattr(bench, "ROOT", str(tmp_path))
        return bench.gemm_source_sha1()

    h0 = digest(base)
    assert digest(dict(base, **{"qgemm.cuh": "// other words\n\nint f(int x) {\n    return x + 1;\n}\n"})) == h0
    assert digest(dict(base, **{"ptx.cuh": "/* changed */\n#pragma once\n"})) == h0
    assert digest(dict(base, **{"qgemm.cuh": "// header\nint f(int x) {\n  return x + 2;  // add\n}\n"})) != h0
