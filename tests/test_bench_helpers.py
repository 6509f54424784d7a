"""bench.py host helpers (no GPU): the DRAM-traffic ratio is read from the committed profile
summary only while the kernel's code matches the capture; the code hash ignores comments
and whitespace but not code; the clocks file path takes the rank."""
import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_ratio_is_read_from_the_summaries(monkeypatch):
    import re
    for wfmt in ("bf16", "mxfp4", "nvfp4"):
        name, files = bench.TRAFFIC[wfmt]
        text = open(os.path.join(ROOT, "profiles", name)).read()
        sha = re.search(r"`kernel_sources_sha256`: `([0-9a-f]{64})`", text).group(1)
        monkeypatch.setattr(bench, "kernel_sources_sha256", lambda f, sha=sha: sha)
        r = bench.traffic_ratio(wfmt)
        assert r is not None and 1.0 <= r < 1.05, (wfmt, r)        # one read per weight byte
    assert bench.traffic_ratio("unknown") is None


def test_traffic_ratio_is_void_once_the_code_changes(monkeypatch):
    monkeypatch.setattr(bench, "kernel_sources_sha256", lambda files: "0" * 64)
    assert bench.traffic_ratio("bf16") is None


def test_code_hash_ignores_comments_and_whitespace(tmp_path, monkeypatch):
    csrc = tmp_path / "expert_cached_sparse_top_b300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cu").write_text("int a = 1; // one\n/* block\n comment */\nint b = 2;\n")
    h0 = bench.kernel_sources_sha256(["k.cu"])
    (csrc / "k.cu").write_text("int  a = 1;   // another comment\n\nint b = 2;  /* x */\n")
    assert bench.kernel_sources_sha256(["k.cu"]) == h0
    (csrc / "k.cu").write_text("int a = 1;\nint b = 3;\n")
    assert bench.kernel_sources_sha256(["k.cu"]) != h0


def test_clocks_path_takes_the_rank():
    a = argparse.Namespace(clocks_csv="out/clocks_r%d.csv")
    assert bench.clocks_path(a, 3) == "out/clocks_r3.csv"
    a = argparse.Namespace(clocks_csv="out/clocks.csv")
    assert bench.clocks_path(a, 3) == "out/clocks.csv"
    a = argparse.Namespace(clocks_csv=None)
    assert bench.clocks_path(a, 1).endswith("ftmoe_clocks_r1.csv")
