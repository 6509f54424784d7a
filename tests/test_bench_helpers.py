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


def test_traffic_summaries_match_the_current_kernels():
    """The committed DRAM-traffic summaries were captured on the kernels as they are now (a
    kernel change voids them: the bench then reports no traffic until they are recaptured)."""
    for wfmt in ("bf16", "mxfp4", "nvfp4"):
        assert bench.traffic_ratio(wfmt) is not None, wfmt


def test_l2_flush_writes_the_whole_buffer_in_every_mode():
    import torch
    for mode in bench.FLUSH_MODES:
        buf = torch.full((4096,), 7, dtype=torch.uint8)
        bench.l2_flush(buf, mode)
        assert int(buf.sum()) == 0
        assert mode in bench.FLUSH_TEXT


def _bench(*args, timeout=240):
    import subprocess
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_warmup_below_three_is_refused():
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "2", timeout=120)
    assert r.returncode != 0 and "--warmup must be >= 3" in r.stderr


def test_reference_arm_prints_the_contract_line():
    """The reference arm is the oracle as it stands, timed on the host cores: one JSON line with
    the headline's metric and unit, an end-to-end block without device copies and a
    cpu_baseline that says what it timed."""
    import json
    r = _bench("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.DECODE[bench.WORKLOAD][0]
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
