"""Host logic of bench.py that needs no GPU: the DRAM-traffic record that
`roofline.traffic` reports is keyed to a hash of the kernel sources, which
must ignore comments and blank space but follow any change of code, and is
reported only while the sources still hash to the recorded value."""
import importlib.util
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_every_hashed_source_exists(bench):
    for f in bench._DRAFT_SOURCES:
        assert os.path.exists(os.path.join(ROOT, "verify_markov_head_gb300", "csrc", f)), f
    assert len(bench._draft_source_hash()) == 16


def test_comments_keep_the_hash_and_code_changes_it(bench):
    code = "__global__ void k(int* x) {\n    x[0] = 1;   // one\n}\n"
    h0 = bench._normalised_source_hash([code])
    assert bench._normalised_source_hash([code + "\n// a comment only\n/* and a block\n   comment */\n\n"]) == h0
    assert bench._normalised_source_hash(["  " + code.replace("\n", "\n\n")]) == h0
    assert bench._normalised_source_hash([code.replace("x[0] = 1", "x[0] = 2")]) != h0
    assert bench._normalised_source_hash([code, code]) != h0


def test_traffic_is_reported_only_for_the_recorded_sources(bench, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    shas = {e["source_sha256"] for k in ("draft_rows", "target_side") for e in [rec[k]["b64"]]}
    assert len(shas) == 1, "the pair's two captures come from the same sources"
    sha = rec["draft_rows"]["b64"]["source_sha256"]
    monkeypatch.setattr(bench, "_draft_source_hash", lambda: sha)
    want = sum(int(rec[k]["b64"]["dram_bytes_per_launch"]) for k in ("draft_rows", "target_side"))
    assert bench._draft_traffic("b64", fused=True) == want
    assert bench._draft_traffic("b64", fused=False) == int(rec["draft_rows"]["b64"]["dram_bytes_per_launch"])
    assert bench._draft_traffic("no-such-workload", fused=True) is None
    monkeypatch.setattr(bench, "_draft_source_hash", lambda: "0" * 16)
    assert bench._draft_traffic("b64", fused=True) is None
