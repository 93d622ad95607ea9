"""Pins for the 12-bit exponent-window format of the oracle.

Format: muse_bf16_proj project report, "Round 5 -- lossless 12-bit
compressed weights", "Format".  Pinned by: exhaustive round trip of every
bf16 bit pattern; the window choice on histograms with a known answer; the
escape rate the pages print (tests/golden/expwin12_escape_rate.json).
"""
import json
import os

import numpy as np
import pytest

from oracle import oracle
from gemv_projection_layers_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("e0", [0, 1, 54, 60, 120])
def test_every_bf16_pattern_round_trips(e0):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    low, nib, esc, esc_hi = oracle.expwin12_encode(bits, e0)
    assert low.dtype == np.uint8 and nib.max() <= 15
    back = oracle.expwin12_decode(low, nib, esc, esc_hi, e0)
    assert np.array_equal(back, bits)
    # exactly the patterns whose 7 high exponent bits leave the window escape
    h7 = (bits >> 8) & 0x7F
    assert esc.size == int(((h7 < e0) | (h7 > e0 + 7)).sum())


def test_low_byte_and_sign_are_stored_raw():
    bits = np.array([0x3C85, 0xBC85, 0x0001, 0x8000], np.uint16)
    low, nib, esc, _ = oracle.expwin12_encode(bits, 54)
    assert low.tolist() == [0x85, 0x85, 0x01, 0x00]
    assert [(n >> 3) for n in nib] == [0, 1, 0, 1]
    assert (0x3C85 >> 8) & 0x7F == 60 and nib[0] & 7 == 6
    assert esc.tolist() == [2, 3]          # zero-exponent patterns escape


def test_window_choice_known_answers():
    def pats(h7_values):
        return (np.asarray(h7_values, np.uint16) << 8)

    assert oracle.expwin12_window(pats([60] * 10)) == 53          # tie -> smallest e0
    assert oracle.expwin12_window(pats([0] * 3 + [1])) == 0
    assert oracle.expwin12_window(pats([127] * 4)) == 120
    # 9 distinct values 40..48: the window can hold 8; both 40..47 and 41..48
    # hold 8 weights when counts are equal -> smallest.
    assert oracle.expwin12_window(pats(list(range(40, 49)))) == 40
    # extra mass at 48 moves the window up by one
    assert oracle.expwin12_window(pats(list(range(40, 49)) + [48])) == 41
    # sign bit must not influence the window
    assert oracle.expwin12_window(pats([60] * 5) | np.uint16(0x8000)) == 53


def test_escape_rate_matches_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "expwin12_escape_rate.json")))
    W = wl.make_weights("pooler", 0)
    e0 = oracle.expwin12_window(W)
    _, _, esc, _ = oracle.expwin12_encode(W, e0)
    pct = 100.0 * esc.size / W.size
    # The pages print "0.014 %" for pooler: read as 0.0135 <= pct < 0.0145.
    assert abs(pct - g["pooler_escape_percent"]) < 0.0005, pct
    assert e0 == 54   # window = magnitudes [2^-19, 2^-3)
    for layer in ("qkv_gate", "o", "unpooler"):
        Wl = wl.make_weights(layer, 1)
        e = oracle.expwin12_window(Wl)
        _, _, es, _ = oracle.expwin12_encode(Wl, e)
        p = 100.0 * es.size / Wl.size
        lo, hi = g["band_percent"]
        # band of the pages, widened by 5 % of its lower end for the K = 4096
        # layer whose N(0, 1/K) spread sits lower than the pooler's
        assert lo * 0.95 <= p <= hi * 1.05, (layer, p)


def test_stream_bytes_ratio():
    g = json.load(open(os.path.join(GOLDEN, "expwin12_escape_rate.json")))
    n = 4096 * 8192
    b = oracle.expwin12_bytes(n, int(n * 0.00014))
    assert abs(b / (2 * n) - g["bytes_ratio"]) < 0.001


def test_stream_bytes_match_the_encoded_fields():
    """The byte count of the format equals what the encoder emits: one low
    byte per weight, two 4-bit nibbles per byte, and a 4-byte entry
    (position, original high byte) per escape."""
    W = wl.make_weights("pooler", 0)
    bits = W.ravel()
    e0 = oracle.expwin12_window(bits)
    low, nib, esc, esc_high = oracle.expwin12_encode(bits, e0)
    assert low.dtype == np.uint8 and low.size == bits.size
    assert int(nib.max()) < 16 and nib.size == bits.size
    packed = (nib[0::2].astype(np.uint16) | (nib[1::2].astype(np.uint16) << 4))
    assert int(packed.max()) < 256 and packed.size == bits.size // 2
    assert esc_high.dtype == np.uint8 and esc_high.size == esc.size
    emitted = low.size + packed.size + 4 * esc.size
    assert emitted == oracle.expwin12_bytes(bits.size, esc.size)
    assert 0.75 < emitted / (2 * bits.size) < 0.7504


@pytest.mark.parametrize("e0", [0, 54, 121])
def test_inband_code7_round_trips_every_pattern(e0):
    """The in-band variant (code 7 marks an escape) is lossless for every
    bf16 pattern, and escapes exactly the patterns outside its 7-wide
    window."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    low, nib, esc_hi = oracle.expwin12_inband_encode(bits, e0)
    assert np.array_equal(oracle.expwin12_inband_decode(low, nib, esc_hi, e0), bits)
    h7 = (bits >> 8) & 0x7F
    assert esc_hi.size == int(((h7 < e0) | (h7 > e0 + 6)).sum())
    assert int(((nib & 7) == 7).sum()) == esc_hi.size


def test_fp32_correction_is_exact_only_near_the_window():
    """The pages' correction term w - w_clamped is an fp32 value when the
    escaped exponent lies at most 14 binades from the window edge (the two
    8-bit significands then span at most 22 bits), and is not one, for an odd
    significand, at 18 binades or more (the span exceeds fp32's 24 bits):
    checked against every bf16 pattern.  The clamped weight keeps the low byte,
    so the exponent distance is twice the high7 distance."""
    e0 = 54
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    _, _, esc, _ = oracle.expwin12_encode(bits, e0)
    exact = oracle.expwin12_correction_exact(bits, e0)
    h7 = ((bits[esc] >> 8) & 0x7F).astype(np.int64)
    gap = np.where(h7 < e0, e0 - h7, h7 - (e0 + 7))
    assert gap.min() == 1
    assert exact[gap <= 7].all()
    zero = (bits[esc] & 0x7FFF) == 0                  # +-0: delta = -w_clamped
    assert exact[zero].all()
    odd = (bits[esc] & 1) == 1
    assert not exact[(gap >= 9) & odd].any()


def test_escape_designs_on_the_layers():
    """Escape designs on the synthetic weights: the in-band window of 7 at
    least doubles the escapes but needs 1 byte each; the position list and
    the in-band code stay below 1.5006 bytes per weight, the bitmap above
    1.515; the pages' correction is exact for every escape of these
    N(0, 1/K) weights."""
    for layer in ("qkv_gate", "o", "pooler", "unpooler"):
        t = oracle.expwin12_variant_table(wl.make_weights(layer, 0))
        assert t["inband_escapes"] >= 2 * t["escapes"], (layer, t)
        assert t["bytes_per_weight"]["position_list"] < 1.5006, (layer, t)
        assert t["bytes_per_weight"]["inband_code7"] < 1.5006, (layer, t)
        assert t["bytes_per_weight"]["bitmap"] > 1.515, (layer, t)
        assert t["fp32_correction_inexact"] == 0, (layer, t)
