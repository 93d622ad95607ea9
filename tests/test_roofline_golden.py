"""Pins for the roofline and score arithmetic against the pages' printed
numbers (muse_bf16_proj guide, ch. 1, §1.7 and §1.8)."""
import json
import os

import pytest

from oracle import roofline
from gemv_projection_layers_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(layer, m):
    return 1024 if (layer.name == "unpooler" and m <= 8) else layer.N


def _load_floor_us(m, bw, peak):
    t = 0.0
    for s in wl.LAYERS:
        rows = _rows(s, m)
        wb = 4 if s.weight_dtype == "fp32" else 2
        ob = 4 if s.out_dtype == "fp32" else 2
        b = roofline.shape_bytes(rows, s.K, m, wb, ob)
        f = roofline.shape_flops(rows, s.K, m)
        t += roofline.floor_seconds(b, f, bw, peak)
    return t * 1e6


def test_per_load_floor_column_is_reproduced():
    g = json.load(open(os.path.join(GOLDEN, "per_load_table.json")))
    bw, peak = g["h200_hbm_bytes_per_s"], g["h200_bf16_flops_per_s"]
    for load, m, sg, ours, floor, sp in g["rows"]:
        assert wl.LOAD_M[load] == m
        assert _load_floor_us(m, bw, peak) == pytest.approx(floor, abs=0.02), load
        assert sg / ours == pytest.approx(sp, abs=0.0015), load


def test_geomean_score():
    g = json.load(open(os.path.join(GOLDEN, "per_load_table.json")))
    sg = [r[2] for r in g["rows"]]
    ours = [r[3] for r in g["rows"]]
    assert roofline.score(sg, ours) == pytest.approx(g["geomean_speedup"], abs=0.0006)


def test_worked_examples():
    e = json.load(open(os.path.join(GOLDEN, "roofline_examples.json")))
    g = json.load(open(os.path.join(GOLDEN, "per_load_table.json")))
    bw, peak = g["h200_hbm_bytes_per_s"], g["h200_bf16_flops_per_s"]
    pooler = wl.LAYER_BY_NAME["pooler"]
    wbytes = pooler.N * pooler.K * 2
    assert wbytes / 1e6 == pytest.approx(e["pooler_m1"]["weight_bytes_MB"], abs=0.05)
    assert wbytes / bw * 1e6 == pytest.approx(e["pooler_m1"]["bytes_us"], abs=0.005)
    f = roofline.shape_flops(pooler.N, pooler.K, 1)
    assert f / 1e6 == pytest.approx(e["pooler_m1"]["mflop"], abs=0.5)
    assert f / peak * 1e6 == pytest.approx(e["pooler_m1"]["math_us"], abs=0.005)
    qkv = wl.LAYER_BY_NAME["qkv_gate"]
    b = roofline.shape_bytes(qkv.N, qkv.K, 16, 2, 2)
    f = roofline.shape_flops(qkv.N, qkv.K, 16)
    assert b / bw * 1e6 == pytest.approx(e["qkv_gate_m16"]["bytes_us"], abs=0.1)
    assert f / 1e9 == pytest.approx(e["qkv_gate_m16"]["gflop"], abs=0.005)
    assert f / peak * 1e6 == pytest.approx(e["qkv_gate_m16"]["math_us"], abs=0.005)
    assert round((b / bw) / (f / peak)) == e["qkv_gate_m16"]["bytes_over_math"]
    # score change when decode 1 drops from 38.25 to 35 us
    sc = e["score_change"]
    sg = [r[2] for r in g["rows"]]
    ours = [r[3] for r in g["rows"]]
    ours2 = [sc["decode1_to_us"] if r[0] == "decode1" else r[3] for r in g["rows"]]
    assert roofline.score(sg, ours) == pytest.approx(sc["score_from"], abs=0.0006)
    assert roofline.score(sg, ours2) == pytest.approx(sc["score_to"], abs=0.001)
