"""Host-side logic of bench.py that needs no GPU: the DRAM-traffic figure the
roofline reports, taken from the committed small-case captures and scaled to
the run's shape, and refused whenever it cannot stand for the run."""

import json
import os

import pytest

import bench


def _write(tmp_path, sha="abc"):
    os.makedirs(tmp_path / "profiles")
    doc = {
        "case": {"T": 16384, "Hd": 2048, "V": 65536, "chunk": 8192},
        "source_sha": sha,
        "kernels": {
            "bwd_dh_dw": {"scale": "V", "first_chunk": {"median": 4.0e9}, "later_chunks": {"median": 5.0e9}},
            "fwd_logits_lse": {"scale": "none", "median": 0.6e9},
        },
    }
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(doc))


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    _write(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "abc")
    return tmp_path


def test_backward_traffic_scales_with_V_and_weights_the_chunks(fake_root):
    # 8 launches per step: one first chunk (dW stored) and 7 later ones (dW reduce-added)
    got = bench.traffic_from_profiles("bwd_dh_dw", 65536, 2048, 124160, chunk=8192, launches_per_step=8)
    assert got == pytest.approx((4.0e9 + 7 * 5.0e9) / 8 * 124160 / 65536)
    assert bench.traffic_from_profiles("bwd_dh_dw", 65536, 2048, 65536, 8192, 1) == pytest.approx(4.0e9)


def test_traffic_is_refused_where_it_does_not_apply(fake_root, monkeypatch):
    assert bench.traffic_from_profiles("bwd_dh_dw", 65536, 2048, 124160, chunk=3968, launches_per_step=17) is None
    assert bench.traffic_from_profiles("bwd_dh_dw", 65536, 4096, 124160, chunk=8192, launches_per_step=8) is None
    assert bench.traffic_from_profiles("bwd_dz", 65536, 2048, 124160, chunk=8192, launches_per_step=8) is None
    # the forward's traffic is not scaled: only the captured shape itself
    assert bench.traffic_from_profiles("fwd_logits_lse", 16384, 2048, 65536) == pytest.approx(0.6e9)
    assert bench.traffic_from_profiles("fwd_logits_lse", 65536, 2048, 124160) is None
    # captures taken on other kernel sources are never reported
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: "def")
    assert bench.traffic_from_profiles("bwd_dh_dw", 65536, 2048, 124160, chunk=8192, launches_per_step=8) is None


def test_committed_traffic_summary_is_well_formed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as fh:
        doc = json.load(fh)
    assert set(doc["case"]) >= {"T", "Hd", "V", "chunk"} and len(doc["source_sha"]) == 16
    for name in ("fwd_logits_lse", "bwd_dz", "bwd_dh_dw"):
        rec = doc["kernels"][name]
        parts = [rec] if rec["scale"] == "none" else [rec["first_chunk"], rec["later_chunks"]]
        for part in parts:
            vals = sorted(c["read"] + c["write"] for c in part["captures"])
            assert len(vals) == 3 and part["min"] == vals[0] and part["median"] == vals[1]
