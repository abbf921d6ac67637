"""The committed ncu summaries of the decode kernel match its current sources (CPU).

`bench.py` reports `roofline.traffic` (DRAM bytes per launch) only when a summary's recorded source
hash equals the sha256 of the decode kernel's sources; these tests keep a kernel change from going
out without re-captured counters, and check that each recorded figure is the workload's
algorithmic KV bytes plus at most 1 % (the partials of the merge, outputs, page-table reads)."""
import re

import pytest

import bench
import pkv_inputs.workloads as W


@pytest.mark.parametrize("cid", sorted(bench.PROFILE_SUMMARY))
def test_profile_hash_matches_current_sources(cid):
    with open(bench.PROFILE_SUMMARY[cid]) as f:
        text = f.read()
    m = re.search(r"kernel sources sha256:\s*([0-9a-f]{64})", text)
    assert m is not None, "the summary records no source hash"
    assert m.group(1) == bench.decode_sources_sha256(), (
        "the decode kernel changed since its DRAM bytes were captured: capture them again")


@pytest.mark.parametrize("cid", sorted(bench.PROFILE_SUMMARY))
def test_profile_traffic_is_the_algorithmic_bytes(cid):
    traffic = bench.ncu_traffic(cid)
    assert traffic is not None
    cfg = W.CONFIGS[cid]
    algo = bench.kv_bytes_layer(W.make_step(cfg, bench.rank_seed(cfg, 0)), False)
    assert algo <= traffic <= algo * 1.01


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    # a comment or blank line does not change the hash; a code line does
    src = tmp_path / "k.cu"
    src.write_text("int a;\n// note\n\nint b;\n")
    monkeypatch.setattr(bench, "DECODE_SOURCES", [str(src)])
    h0 = bench.decode_sources_sha256()
    src.write_text("int a;\n   // another note\nint b;\n\n")
    assert bench.decode_sources_sha256() == h0
    src.write_text("int a;\nint c;\n")
    assert bench.decode_sources_sha256() != h0
