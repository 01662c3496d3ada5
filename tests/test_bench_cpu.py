"""bench.py's host-side accounting, without a GPU: the algorithmic bytes behind the decode
roofline, the stage that roofline is taken on, and the guard that keeps a recorded ncu
traffic figure tied to the kernel source it was measured on."""
import hashlib

import pytest

import bench
from latent_moe_layer_gb300 import synth

# one expert's record as shipped: w1 and w3 [3072, 3584] and w2 [3584, 3072], MXFP4 (two
# codes per byte plus one E8M0 byte per 32 values) -- 33,030,144 values, 17,547,264 bytes
RECORD_BYTES = 17_547_264


def test_decode_expert_bytes_are_the_touched_records():
    cfg = synth.CONFIGS[1]
    touched = 223
    w = bench.stage_work(cfg, touched, path_tensor=True)
    R = cfg.T * cfg.K
    act_up = R * cfg.L * 2 + R * cfg.I * 2              # f16 expert inputs in, GLU output out
    act_down = R * cfg.I * 2 + R * cfg.L * 2            # GLU output in, expert outputs out
    assert w["gate_up"][0] - act_up == touched * 11_698_176
    assert w["expert_down"][0] - act_down == touched * 5_849_088
    assert (w["gate_up"][0] - act_up + w["expert_down"][0] - act_down) == touched * RECORD_BYTES
    assert w["gate_up"][1] == 4 * R * cfg.I * cfg.L and w["expert_down"][1] == 2 * R * cfg.L * cfg.I


def test_fused_decode_launch_counts_both_projections():
    w = {"gate_up": (10, 1), "expert_down": (5, 2), "router": (3, 0)}
    dom, (b, f), fused = bench.dominant_stage({"gate_up": 0.6, "router": 0.02}, w)
    assert (dom, b, f, fused) == ("gate_up", 15, 3, True)
    dom, (b, f), fused = bench.dominant_stage({"gate_up": 0.4, "expert_down": 0.2, "router": 0.02}, w)
    assert (dom, b, f, fused) == ("gate_up", 10, 1, False)
    assert w["gate_up"] == (10, 1)                       # the caller's table is not modified


def test_traffic_figure_needs_the_measured_source(tmp_path, monkeypatch):
    src, hdr = tmp_path / "kernel.cu", tmp_path / "kernel.cuh"
    src.write_bytes(b"#include \"kernel.cuh\"\n__global__ void k() {}\n")
    hdr.write_bytes(b"#define W 1\n")
    sha = hashlib.sha256(src.read_bytes() + hdr.read_bytes()).hexdigest()[:16]
    rec = {"sources": [str(src), str(hdr)], "sha256_16": sha, "per_expert": {("gate_up", "gemv"): 1.0}}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", rec)
    monkeypatch.setattr(bench, "ROOT", "/")
    assert bench.ncu_traffic_per_expert() == {("gate_up", "gemv"): 1.0}
    hdr.write_bytes(b"#define W 2\n")                  # an edit of a header the kernel includes
    assert bench.ncu_traffic_per_expert() == {}
    hdr.write_bytes(b"#define W 1\n")
    assert bench.ncu_traffic_per_expert() == {("gate_up", "gemv"): 1.0}
    src.write_bytes(b"#include \"kernel.cuh\"\n__global__ void k() { }\n")   # or of the kernel itself
    assert bench.ncu_traffic_per_expert() == {}
