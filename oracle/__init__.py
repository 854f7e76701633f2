"""f64 CPU oracle for causal prefill attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or calls it, and this
package imports nothing from the product package.

The arithmetic lives in ``fa_oracle.c`` (plain C, IEEE double, libm ``exp``,
compiled with ``-O2`` and no fast-math).  It computes the plain definition

    O = softmax(scale * Q K^T + causal mask) V

row by row over the full score row, with the bottom-right causal alignment
(query row i of Sq sees key j iff j <= (Skv - Sq) + i), the contiguous GQA
grouping hk = hq // (Hq // Hkv), and O = 0 for a row that sees no key.  The
passages each step follows are cited in the C file's header:
minfer "28 · r23 — f16-path whole-graph wall decomposition + FA_TKV occupancy
raise", section 3.2 (the mask), and minfer "53 · r50 — FA_TKV 32->16 occupancy
experiment", sections 2 and 3.2 (the online softmax it stands in for, the
fully-masked-row guard, the KV-head index).

Pins (closed forms, invariants, brute force, a library cross-check) are in
``tests/test_oracle_pins.py``; none of them calls this package to produce an
expected value.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``fa_oracle.c`` into ``liboracle.so`` beside it (gcc, -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d = ctypes.POINTER(ctypes.c_double)
            i32 = ctypes.c_int
            lib.oracle_attention.argtypes = [d, d, d, d] + [i32] * 7 + [ctypes.c_double, i32]
            lib.oracle_attention.restype = i32
            lib.oracle_attention_rows.argtypes = ([d, d, d] + [i32] * 7 + [ctypes.c_double]
                                                  + [ctypes.POINTER(ctypes.c_int32),
                                                     ctypes.c_longlong, d, i32])
            lib.oracle_attention_rows.restype = i32
            lib.oracle_probs_row.argtypes = [d, d] + [i32] * 7 + [ctypes.c_double] + [i32] * 3 + [d]
            lib.oracle_probs_row.restype = i32
            lib.oracle_plant_mistake.argtypes = [i32]
            lib.oracle_plant_mistake.restype = i32
            lib.oracle_round_f16.argtypes = [ctypes.c_float]
            lib.oracle_round_f16.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [ctypes.c_float]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_kv_append.argtypes = ([ctypes.c_void_p] * 5 + [i32] * 6)
            lib.oracle_kv_append.restype = ctypes.c_longlong
            lib.oracle_lse_rows.argtypes = ([d, d] + [i32] * 7 + [ctypes.c_double]
                                            + [ctypes.POINTER(ctypes.c_int32), ctypes.c_longlong, d])
            lib.oracle_lse_rows.restype = i32
            _lib = lib
    return _lib


# Deliberately wrong variants of the oracle, switched on only by the pin tests
# to show that the pins reject them (0 is the correct oracle).
PLANTED_MISTAKES = {
    "none": 0, "no_scale": 1, "top_left": 2, "mask_off_by_one": 3, "gqa_modulo": 4,
    "no_normalise": 5, "v_reversed": 6, "no_max_subtract": 7, "exp2": 8, "masked_row_nan": 9,
    "round_truncate": 10, "round_ties_away": 11, "append_at_t": 12, "lse_log2": 13,
    "gather_swapped": 14, "gather_no_table": 15,
}
# mistakes planted in this file's own arithmetic (the paged gather) rather than in the C library
_PY_PLANTS = ("gather_swapped", "gather_no_table")
_py_plant = "none"


def plant_mistake(kind: str) -> None:
    """Switch the oracle to one planted mistake (``"none"`` restores it). Tests only."""
    global _py_plant
    code = PLANTED_MISTAKES[kind]
    rc = _load().oracle_plant_mistake(0 if kind in _PY_PLANTS else code)
    if rc != 0:
        raise ValueError(kind)
    _py_plant = kind if kind in _PY_PLANTS else "none"


def _f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor or array-like to contiguous float64."""
    if hasattr(x, "detach"):  # torch tensor: f16/bf16 -> f64 is exact
        x = x.detach().to("cpu").double().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _shape(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, S, H, hd]")
    B, Sq, Hq, hd = q.shape
    Bk, Skv, Hkv, hdk = k.shape
    if (Bk, hdk) != (B, hd) or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    return B, Hq, Hkv, Sq, Skv, hd


def attention(q, k, v, causal: bool = True, scale: float | None = None,
              nthreads: int | None = None) -> np.ndarray:
    """Full f64 output [B, Sq, Hq, hd] of softmax(scale QK^T + mask) V."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Skv, hd = _shape(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(hd)
    o = np.zeros((B, Sq, Hq, hd), dtype=np.float64)
    rc = _load().oracle_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, Sq, Skv, hd,
                                  int(bool(causal)), float(scale),
                                  int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention failed with status {rc}")
    return o


def attention_rows(q, k, v, rows, causal: bool = True, scale: float | None = None,
                   nthreads: int | None = None) -> np.ndarray:
    """Selected output rows. ``rows`` is an int array [n, 3] of (b, hq, i); returns [n, hd]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Skv, hd = _shape(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(hd)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    out = np.zeros((r.shape[0], hd), dtype=np.float64)
    rc = _load().oracle_attention_rows(
        _ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Skv, hd, int(bool(causal)), float(scale),
        r.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), r.shape[0], _ptr(out),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed with status {rc}")
    return out


def probs_row(q, k, b: int, hq: int, i: int, causal: bool = True,
              scale: float | None = None) -> np.ndarray:
    """The probability row P[b, hq, i, :] over all Skv keys."""
    q, k = _f64(q), _f64(k)
    B, Hq, Hkv, Sq, Skv, hd = _shape(q, k, k)
    if scale is None:
        scale = 1.0 / np.sqrt(hd)
    p = np.zeros((Skv,), dtype=np.float64)
    rc = _load().oracle_probs_row(_ptr(q), _ptr(k), B, Hq, Hkv, Sq, Skv, hd,
                                  int(bool(causal)), float(scale), b, hq, i, _ptr(p))
    if rc != 0:
        raise ValueError(f"oracle_probs_row failed with status {rc}")
    return p


def round16_bits(x, bf16: bool) -> np.ndarray:
    """IEEE round-to-nearest-even of float32 values into binary16 (bf16=False)
    or bfloat16 (bf16=True); returns the 16-bit patterns as uint16."""
    lib = _load()
    f = lib.oracle_round_bf16 if bf16 else lib.oracle_round_f16
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).ravel()
    out = np.empty(a.shape, dtype=np.uint16)
    for i, v in enumerate(a.tolist()):
        out[i] = f(v)
    return out.reshape(np.shape(x))


def kv_append(k_new, v_new, positions, k_cache_bits, v_cache_bits, bf16: bool):
    """The K/V-cache append on numpy arrays: k_new, v_new float32 [B][T][Hkv][hd];
    positions int32 [B][T]; caches uint16 bit patterns [B][cap][Hkv][hd],
    updated in place.  Returns the number of tokens skipped (position out of range)."""
    kn = np.ascontiguousarray(k_new, dtype=np.float32)
    vn = np.ascontiguousarray(v_new, dtype=np.float32)
    ps = np.ascontiguousarray(positions, dtype=np.int32)
    for c in (k_cache_bits, v_cache_bits):
        if c.dtype != np.uint16 or not c.flags.c_contiguous:
            raise ValueError("caches must be contiguous uint16 arrays")
    B, T, Hkv, hd = kn.shape
    cap = k_cache_bits.shape[1]
    n = _load().oracle_kv_append(kn.ctypes.data, vn.ctypes.data, ps.ctypes.data, k_cache_bits.ctypes.data,
                                 v_cache_bits.ctypes.data, B, T, Hkv, hd, cap, int(bool(bf16)))
    if n < 0:
        raise ValueError("bad arguments")
    return int(n)


def gather_pages(pool, block_table, kv_len: int, page_size: int):
    """Contiguous K or V [B, kv_len, Hkv, hd] from a paged pool
    [num_blocks, page_size, Hkv, hd] and a block table [B, max_pages]: key j
    of sequence b is pool[block_table[b, j // page_size], j % page_size] (the
    definition of a paged cache; the attention oracle then runs on the result)."""
    pool = np.asarray(pool.detach().cpu().double().numpy() if hasattr(pool, "detach") else pool, dtype=np.float64)
    table = np.asarray(block_table.cpu().numpy() if hasattr(block_table, "cpu") else block_table, dtype=np.int64)
    j = np.arange(kv_len)
    page, row = j // page_size, j % page_size
    if _py_plant == "gather_swapped":  # planted mistake: page and row index exchanged
        page, row = row, page
    if _py_plant == "gather_no_table":  # planted mistake: the page number used as the pool block
        return np.ascontiguousarray(np.broadcast_to(pool[page, row], (table.shape[0],) + pool[page, row].shape))
    return np.ascontiguousarray(pool[table[:, page], row])


def lse_rows(q, k, rows, causal: bool = True, scale: float | None = None) -> np.ndarray:
    """Per-row log-sum-exp of the scaled, masked scores for rows [n, 3] =
    (b, hq, i): log sum_j exp(s_j) over the visible keys, -inf for a row that
    sees none.  Returns float64 [n]."""
    qa, ka = _f64(q), _f64(k)
    B, Sq, Hq, hd = qa.shape
    _, Skv, Hkv, _ = ka.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(hd))
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    out = np.empty(r.shape[0], dtype=np.float64)
    rc = _load().oracle_lse_rows(_ptr(qa), _ptr(ka), B, Hq, Hkv, Sq, Skv, hd, int(bool(causal)), float(scale),
                                 r.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), r.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_lse_rows failed ({rc})")
    return out


def lse(q, k, causal: bool = True, scale: float | None = None) -> np.ndarray:
    """log-sum-exp of every row, as [B, Hq, Sq] float64."""
    qa = _f64(q)
    B, Sq, Hq, _ = qa.shape
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(Sq), indexing="ij")
    rows = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    return lse_rows(q, k, rows, causal, scale).reshape(B, Hq, Sq)
