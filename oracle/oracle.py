"""Oracle for the dense projection path -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this module.  It shares no code with the CUDA path (the two meet only
in the seeded input generators of gemv_projection_layers_gb300.workloads).

Contents, each restated from the pages:

* reference(): FP64 dot products, out = x @ W.T -- plain C in proj_oracle.c
  (muse_bf16_proj guide, ch. 1, §1.1 "What is computed").
* out_rows(): the unpooler computes only its first 1024 rows at <= 8 tokens
  (guide ch. 1, §1.1 table, unpooler row).
* check(): the correctness contract of guide ch. 1, §1.5 "What counts as
  correct" -- relative L2 per output tensor <= 1 % (router 0.01 %), probe rows
  within 0.1 %, no row over 5x the bound, no NaN/Inf.
* expwin12_inband_*, expwin12_correction_exact, expwin12_variant_table:
  the escape designs compared (in-band code 7; the pages' fp32 correction).
* expwin12_*: the lossless 12-bit exponent-window weight format of the
  project report, "Round 5 -- lossless 12-bit compressed weights", "Format":
  raw low byte + 4-bit (sign, 3-bit window code) + escape list, window of 8
  consecutive values of the 7 high exponent bits chosen per matrix to cover
  the most weights.  Escapes store the original high byte (reading of the
  pages: restore the exact bits before the multiply, instead of the pages'
  fp32 correction term, so that decode(encode(w)) == w for every pattern).

Readings of points the pages leave open (also listed in the design notes):
  - "relative L2 per output" = Frobenius ratio over the whole [m, N] output;
    the 5x rule and the probe rule apply per token row of the output; a row
    whose reference norm is zero is judged by its absolute L2 norm;
  - window tie-break: the smallest e0 in [0, 120] with the maximal count.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "proj_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile proj_oracle.c with gcc (-O2, OpenMP, no FP contraction)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_proj_bf16.argtypes = [p, p, i64, i64, i64, p]
            lib.oracle_proj_f32w.argtypes = [p, p, i64, i64, i64, p]
            lib.oracle_proj_entries.argtypes = [p, p, ctypes.c_int, i64, p, p, i64, p]
            lib.oracle_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def threads() -> int:
    return int(_load().oracle_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


# ---------------------------------------------------------------------------
# The projection
# ---------------------------------------------------------------------------

ROUTER = "router"


def out_rows(layer: str, N: int, m: int) -> int:
    """Rows of W computed at m tokens (guide ch. 1, §1.1: unpooler slice)."""
    if layer == "unpooler" and m <= 8:
        return 1024
    return N


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def reference(layer: str, x_bits: np.ndarray, W: np.ndarray) -> np.ndarray:
    """FP64 reference [m, out_rows] for x (bf16 bits [m, K]) and W.

    W is bf16 bits (uint16 [N, K]) for the dense layers and float32 [N, K]
    for the router."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    m, K = x.shape
    N, K2 = W.shape
    if K != K2:
        raise ValueError("x and W disagree on K")
    rows = out_rows(layer, N, m)
    ref = np.empty((m, rows), dtype=np.float64)
    if m == 0:
        return ref
    if W.dtype == np.float32:
        Wc = np.ascontiguousarray(W)
        lib.oracle_proj_f32w(_ptr(x), _ptr(Wc), m, rows, K, _ptr(ref))
    elif W.dtype == np.uint16:
        Wc = np.ascontiguousarray(W)
        lib.oracle_proj_bf16(_ptr(x), _ptr(Wc), m, rows, K, _ptr(ref))
    else:
        raise TypeError("W must be uint16 (bf16 bits) or float32")
    return ref


def reference_entries(x_bits: np.ndarray, W: np.ndarray, rows_i, rows_n) -> np.ndarray:
    """FP64 reference of selected outputs ref[rows_i[j], rows_n[j]]."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ri = np.ascontiguousarray(rows_i, dtype=np.int64)
    rn = np.ascontiguousarray(rows_n, dtype=np.int64)
    out = np.empty(ri.shape[0], dtype=np.float64)
    Wc = np.ascontiguousarray(W)
    lib.oracle_proj_entries(_ptr(x), _ptr(Wc), int(W.dtype == np.float32), x.shape[1],
                            _ptr(ri), _ptr(rn), ri.shape[0], _ptr(out))
    return out


# ---------------------------------------------------------------------------
# Correctness contract (guide ch. 1, §1.5)
# ---------------------------------------------------------------------------

DENSE_TOL = 1e-2
ROUTER_TOL = 1e-4
PROBE_TOL = 1e-3
ROW_FACTOR = 5.0


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def check(layer: str, out: np.ndarray, ref: np.ndarray, probe_rows=()) -> dict:
    """Apply the contract to a device result `out` (float array, any width).

    Returns a dict with the measured figures and `ok`."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if out.shape != ref.shape:
        return {"ok": False, "reason": f"shape {out.shape} != {ref.shape}"}
    tol = ROUTER_TOL if layer == ROUTER else DENSE_TOL
    finite = bool(np.isfinite(out).all())
    diff = out - ref
    ref_norm = float(np.sqrt((ref * ref).sum()))
    err_norm = float(np.sqrt((diff * diff).sum()))
    rel = err_norm / ref_norm if ref_norm > 0 else err_norm
    row_ref = np.sqrt((ref * ref).sum(axis=1))
    row_err = np.sqrt((diff * diff).sum(axis=1))
    row_rel = np.where(row_ref > 0, row_err / np.where(row_ref > 0, row_ref, 1.0), row_err)
    worst_row = float(row_rel.max()) if row_rel.size else 0.0
    probe = [int(r) for r in probe_rows]
    probe_rel = float(row_rel[probe].max()) if probe else 0.0
    ok = (finite and rel <= tol and worst_row <= ROW_FACTOR * tol
          and probe_rel <= PROBE_TOL)
    return {"ok": bool(ok), "finite": finite, "rel_l2": rel, "tol": tol,
            "worst_row_rel": worst_row, "row_bound": ROW_FACTOR * tol,
            "probe_rel": probe_rel, "probe_tol": PROBE_TOL}


# ---------------------------------------------------------------------------
# 12-bit exponent-window format (project report, Round 5, "Format")
# ---------------------------------------------------------------------------

EXPWIN_SPAN = 8          # 3-bit code -> 8 consecutive values
EXPWIN_E0_MAX = 127 - 7  # keeps e0 + 7 within the 7-bit field


def expwin12_high7(bits: np.ndarray) -> np.ndarray:
    """The 7 high exponent bits of each bf16 pattern (bits 14..8)."""
    return (np.asarray(bits, dtype=np.uint16) >> 8).astype(np.int64) & 0x7F


def expwin12_window(bits: np.ndarray) -> int:
    """e0 in [0, 120] maximising #weights with high7 in [e0, e0 + 7]
    (smallest e0 on a tie)."""
    hist = np.bincount(expwin12_high7(bits).ravel(), minlength=128)
    best_e0, best = 0, -1
    for e0 in range(EXPWIN_E0_MAX + 1):
        c = int(hist[e0:e0 + EXPWIN_SPAN].sum())
        if c > best:
            best_e0, best = e0, c
    return best_e0


def expwin12_encode(bits: np.ndarray, e0: int):
    """Encode bf16 patterns (any shape) with window base e0.

    Returns (low_byte uint8, nibble uint8 in [0, 15], esc_index int64,
    esc_high uint8): nibble = sign << 3 | code, code = clamp(high7 - e0, 0, 7);
    escapes are the flat indices whose high7 lies outside the window, with
    their original high byte (sign + high7)."""
    b = np.asarray(bits, dtype=np.uint16).ravel()
    low = (b & 0xFF).astype(np.uint8)
    sign = (b >> 15).astype(np.int64)
    h7 = (b.astype(np.int64) >> 8) & 0x7F
    code = np.clip(h7 - e0, 0, EXPWIN_SPAN - 1)
    nib = ((sign << 3) | code).astype(np.uint8)
    esc = np.flatnonzero((h7 < e0) | (h7 > e0 + EXPWIN_SPAN - 1)).astype(np.int64)
    esc_high = (b[esc] >> 8).astype(np.uint8)
    return low, nib, esc, esc_high


def expwin12_decode(low: np.ndarray, nib: np.ndarray, esc_index: np.ndarray,
                    esc_high: np.ndarray, e0: int) -> np.ndarray:
    """Inverse of expwin12_encode (flat uint16 bf16 patterns)."""
    n = nib.astype(np.uint16)
    high = ((n >> 3) << 7) | (np.uint16(e0) + (n & 7))
    high = high.astype(np.uint16)
    high[esc_index] = esc_high.astype(np.uint16)
    return ((high << 8) | low.astype(np.uint16)).astype(np.uint16)


def expwin12_bytes(n_weights: int, n_escapes: int, escape_entry_bytes: int = 4) -> int:
    """Stream bytes of the format: 1.5 bytes per weight plus the escapes."""
    return (n_weights * 3) // 2 + n_escapes * escape_entry_bytes


# --- escape designs compared (project report, "Round 5", "Format" and
# "Kernel": the exception list; the alternatives the design notes weigh) ---

def expwin12_inband_window(bits: np.ndarray) -> int:
    """In-band variant: e0 maximising #weights with high7 in [e0, e0 + 6]
    (code 7 is reserved to mark an escape; smallest e0 on a tie)."""
    hist = np.bincount(expwin12_high7(bits).ravel(), minlength=128)
    best_e0, best = 0, -1
    for e0 in range(127 - 6 + 1):
        c = int(hist[e0:e0 + EXPWIN_SPAN - 1].sum())
        if c > best:
            best_e0, best = e0, c
    return best_e0


def expwin12_inband_encode(bits: np.ndarray, e0: int):
    """In-band variant: nibble = sign << 3 | code, code = high7 - e0 in 0..6
    for weights inside the window and 7 for every other weight, whose
    original high byte goes, in stream order, to the escape list (its
    position is implied by the code).  Returns (low, nibble, esc_high)."""
    b = np.asarray(bits, dtype=np.uint16).ravel()
    low = (b & 0xFF).astype(np.uint8)
    sign = (b >> 15).astype(np.int64)
    h7 = (b.astype(np.int64) >> 8) & 0x7F
    inside = (h7 >= e0) & (h7 <= e0 + EXPWIN_SPAN - 2)
    code = np.where(inside, h7 - e0, EXPWIN_SPAN - 1)
    nib = ((sign << 3) | code).astype(np.uint8)
    esc_high = (b[~inside] >> 8).astype(np.uint8)
    return low, nib, esc_high


def expwin12_inband_decode(low: np.ndarray, nib: np.ndarray, esc_high: np.ndarray,
                           e0: int) -> np.ndarray:
    """Inverse of expwin12_inband_encode (flat uint16 bf16 patterns)."""
    n = nib.astype(np.uint16)
    code = n & 7
    high = (((n >> 3) << 7) | (np.uint16(e0) + code)).astype(np.uint16)
    esc = code == EXPWIN_SPAN - 1
    high[esc] = esc_high.astype(np.uint16)
    return ((high << 8) | low.astype(np.uint16)).astype(np.uint16)


def expwin12_correction_exact(bits: np.ndarray, e0: int) -> np.ndarray:
    """The pages' exception design: an escaped weight is stored with its
    exponent clamped into the window and corrected by an fp32 term
    delta = w - w_clamped.  True where that delta is exactly an fp32 value
    (so w_clamped + delta reproduces w), per escaped weight of
    expwin12_encode (in its order).  The difference is taken in rationals
    (an FP64 subtraction would itself round when the two are more than 45
    binades apart); +-inf counts as exact, NaN as not."""
    from fractions import Fraction
    b = np.asarray(bits, dtype=np.uint16).ravel()
    _, nib, esc, _ = expwin12_encode(b, e0)
    n16 = nib.astype(np.uint16)
    clamped = (((n16 >> 3) << 15) | ((np.uint16(e0) + (n16 & 7)) << 8) |
               (b & 0xFF)).astype(np.uint16)
    w = bf16_bits_to_f64(b[esc])
    wc = bf16_bits_to_f64(clamped[esc])
    out = np.zeros(esc.size, dtype=bool)
    for i in range(esc.size):
        if np.isinf(w[i]):
            out[i] = True
        elif np.isfinite(w[i]):
            d = Fraction(float(w[i])) - Fraction(float(wc[i]))
            out[i] = Fraction(float(np.float32(float(d)))) == d
    return out


def expwin12_variant_table(bits: np.ndarray) -> dict:
    """Escapes and stream bytes per weight of four escape designs on one
    matrix: the position list (1.5 B + a 4-byte (position, high byte) entry
    per escape), the in-band code 7 (1.5 B + the 1-byte high byte per
    escape, window of 7), a bitmap (1.5 B + 1 bit per 8 weights + 2 bytes
    per escape: in-group position and high byte) and the pages' fp32
    correction (1.5 B + 8 bytes per escape: position and fp32 delta), with
    the correction's inexact escapes."""
    b = np.asarray(bits, dtype=np.uint16).ravel()
    n = b.size
    e0 = expwin12_window(b)
    _, _, esc, _ = expwin12_encode(b, e0)
    e7 = expwin12_inband_window(b)
    _, _, esc7 = expwin12_inband_encode(b, e7)
    exact = expwin12_correction_exact(b, e0)
    k = esc.size
    return {
        "weights": n,
        "window_e0": e0, "escapes": k, "escape_percent": 100.0 * k / n,
        "groups_of_8_with_escape_percent": 100.0 * np.unique(esc // 8).size / (n // 8),
        "inband_window_e0": e7, "inband_escapes": int(esc7.size),
        "inband_escape_percent": 100.0 * esc7.size / n,
        "bytes_per_weight": {
            "position_list": (1.5 * n + 4 * k) / n,
            "inband_code7": (1.5 * n + 1 * esc7.size) / n,
            "bitmap": (1.5 * n + n / 64 + 2 * k) / n,
            "fp32_correction": (1.5 * n + 8 * k) / n,
        },
        "fp32_correction_inexact": int((~exact).sum()),
    }
