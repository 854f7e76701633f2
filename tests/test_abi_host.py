"""The C ABI on the host, no GPU needed: the library builds and loads, exports
every symbol include/fa_prefill.h declares, and rejects bad arguments before
touching a device (resource and argument errors fail loudly -- minfer "11 · P5
— prefill gap session: TM=128 big tiles + FA rewrite", section 3.3)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_prefill.h")


@pytest.fixture(scope="module")
def fa():
    import causal_prefill_flash_gb300 as fa
    fa.build()
    fa.load()
    return fa


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_prefill", "fa_prefill_bf16", "fa_prefill_ws", "fa_prefill_ws_bf16", "fa_workspace_bytes",
              "fa_status_string", "fa_smem_bytes", "fa_debug_status", "fa_debug_status_clear"):
        assert n in names


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(fa):
    for code, name in fa._lib.STATUS_NAMES.items():
        assert fa.status_string(code).startswith(name)
    assert fa.status_string(99) == "unknown fa_status_t"


def test_smem_request_matches_the_tile_layout(fa):
    """Two query tiles + a ring of K/V slots (5 at hd = 128, 8 at hd = 64) +
    the mbarriers + 16 B of flags + 1 KB alignment slack; within the 227 KB
    opt-in limit.  hd 128: one for Q, a full/empty pair per slot, two each
    for S ready and P ready, the final O and the abort drain (each warp sends
    its own rows of O, so no O-staged barrier).  hd 64: one for Q, 4 (V, K)
    pair barriers, 8 slot frees, two each for S ready, S read, P ready and
    P V done, the final O, the drain, two O-staged."""
    for hd, nslot, bars in ((64, 8, 1 + 4 + 8 + 2 * 4 + 1 + 1 + 2), (128, 5, 1 + 2 * 5 + 2 + 2 + 2)):
        q = 128 * hd * 2
        slot = 128 * hd * 2
        want = 2 * q + nslot * slot + bars * 8 + 16 + 1024
        assert fa.smem_bytes(hd) == want
        assert want <= 227 * 1024
    assert fa.smem_bytes(100) == 0 and fa.smem_bytes(264) == 0
    # narrower heads run on the next kernel up (64, 128 or 256)
    assert fa.smem_bytes(32) == fa.smem_bytes(64) and fa.smem_bytes(96) == fa.smem_bytes(128)
    assert fa.smem_bytes(192) == fa.smem_bytes(256)
    # hd 256: one 64 KB query tile, a ring of five 32 KB half tiles, 18 barriers
    assert fa.smem_bytes(256) == 64 * 1024 + 5 * 32 * 1024 + 18 * 8 + 16 + 1024 <= 227 * 1024


A = 0x10000  # aligned fake device addresses: validation fails before any use


@pytest.mark.parametrize("fn", ["fa_prefill", "fa_prefill_bf16"])
def test_argument_errors_without_a_device(fa, fn):
    f = getattr(fa, fn)
    ok = dict(q=A, k=2 * A, v=3 * A, o=4 * A, B=1, Hq=4, Hkv=2, Sq=8, Skv=8, hd=128, causal=1, scale=0.1)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["hd"],
                 a["causal"], a["scale"], 0)

    assert call(q=0) == 1 and call(o=0) == 1 and call(k=0) == 1 and call(v=0) == 1
    assert call(Skv=0, k=0, v=0, hd=100) == 2  # shape errors still reported first
    assert call(B=-1) == 1 and call(Sq=-3) == 1 and call(Skv=-1) == 1
    assert call(Hq=0) == 1 and call(Hkv=0) == 1 and call(Hkv=3) == 1
    assert call(scale=float("nan")) == 1 and call(scale=0.0) == 1 and call(scale=-1.0) == 1
    # hd: a multiple of 8 (16-byte rows) up to 256
    assert call(hd=100) == 2 and call(hd=512) == 2 and call(hd=4) == 2 and call(hd=264) == 2 and call(hd=0) == 2
    assert call(q=A + 8) == 3 and call(o=4 * A + 2) == 3
    assert call(o=A) == 1  # o overlaps q
    assert call(Sq=2 ** 31 - 100) == 2
    # nothing to compute: FA_OK without a device, null pointers allowed
    assert call(B=0) == 0 and call(Sq=0) == 0
    assert call(B=0, q=0, k=0, v=0, o=0) == 0 and call(Sq=0, q=0, o=0) == 0


def test_python_wrapper_rejects_cpu_tensors(fa):
    import torch
    q = torch.zeros((1, 4, 2, 128), dtype=torch.float16)
    with pytest.raises(ValueError):
        fa.attention(q, q, q)


def test_workspace_size_and_errors_without_a_device(fa):
    """Stream-K workspace: 512 piece slots (a CTA of up to 256 holds at most two
    pieces of split pairs), each with both tiles' partial O in f32 and m and l
    per row."""
    for hd in (64, 128):
        o_bytes = 512 * 2 * 128 * hd * 4
        ml_bytes = 512 * 2 * 2 * 128 * 4
        assert fa.workspace_bytes(hd) == o_bytes + ml_bytes
    for hd, kh in ((8, 64), (40, 64), (72, 128), (80, 128), (96, 128), (120, 128)):
        assert fa.workspace_bytes(hd) == fa.workspace_bytes(kh)  # runs on the next kernel up
    assert fa.workspace_bytes(84) == 0 and fa.workspace_bytes(192) == 0 and fa.workspace_bytes(256) == 0
    ws = fa.workspace_bytes(128)
    args = (A, 2 * A, 3 * A, 4 * A, 1, 4, 2, 8, 8, 128, 1, 0.1)
    for f in (fa.fa_prefill_ws, fa.fa_prefill_ws_bf16):
        assert f(*args, 0, ws, 0) == 1                # no workspace
        assert f(*args, 5 * A + 16, ws, 0) == 3       # not 256-byte aligned
        assert f(*args, 5 * A, ws - 1, 0) == 1        # too small
        assert f(A, 2 * A, 3 * A, 4 * A, 0, 4, 2, 8, 8, 128, 1, 0.1, 0, 0, 0) == 0  # empty problem: no-op
        assert f(A, 2 * A, 3 * A, 4 * A, 1, 4, 2, 8, 8, 100, 1, 0.1, 5 * A, ws, 0) == 2
        assert f(A, 2 * A, 3 * A, 4 * A, 1, 4, 2, 8, 8, 192, 1, 0.1, 5 * A, ws, 0) == 2  # split-KV: heads up to 128


def test_static_scratch_entry_point_errors_without_a_device(fa):
    """fa_prefill_ws_static checks its arguments like fa_prefill before any
    device call (and before its one-time set-up)."""
    f = fa.fa_prefill_ws_static
    for bf16 in (0, 1):
        args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, B=1, Hq=4, Hkv=2, Sq=8, Skv=8, hd=128, causal=1, scale=0.1)

        def call(**kw):
            a = dict(args, **kw)
            return f(a["q"], a["k"], a["v"], a["o"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Skv"], a["hd"],
                     a["causal"], a["scale"], bf16, 0)

        assert call(q=0) == 1 and call(Hkv=3) == 1 and call(scale=0.0) == 1
        assert call(hd=100) == 2 and call(hd=192) == 2 and call(q=A + 8) == 3
        assert call(B=0) == 0 and call(Sq=0, q=0, o=0) == 0
    assert fa.status_string(7).startswith("FA_ERR_SCRATCH")


def test_split_advice_rejects_bad_sizes_without_a_device(fa):
    f = fa._lib.load().fa_split_kv_advised
    assert f(1, 3, 2, 8, 8, 1) == -1      # Hq % Hkv != 0
    assert f(-1, 4, 2, 8, 8, 1) == -1
    assert f(0, 4, 2, 8, 8, 1) == 0       # nothing to compute: no advice needed, no device touched
    assert f(1, 4, 2, 8, 0, 1) == 0
    g = fa._lib.load().fa_split_kv_advised_hd
    assert g(1, 3, 2, 8, 8, 64, 1) == -1     # Hq % Hkv != 0
    assert g(1, 4, 2, 8, 8, 100, 1) == -2    # no kernel takes hd 100
    assert g(0, 4, 2, 8, 8, 64, 1) == 0
    assert g(1, 4, 2, 8, 8, 256, 1) == 0     # split-KV takes heads up to 128 wide


def test_kvcache_and_append_errors_without_a_device(fa):
    """The cache entry points check their arguments before any device call."""
    ap = fa.fa_kv_append
    ok = dict(kn=A, vn=2 * A, pos=3 * A, kc=4 * A, vc=5 * A, B=1, T=4, Hkv=2, hd=128, cap=16, bf16=0)

    def append(**kw):
        a = dict(ok, **kw)
        return ap(a["kn"], a["vn"], a["pos"], a["kc"], a["vc"], a["B"], a["T"], a["Hkv"], a["hd"], a["cap"],
                  a["bf16"], 0)

    assert append(kn=0) == 1 and append(pos=0) == 1 and append(vc=0) == 1
    assert append(B=-1) == 1 and append(T=-1) == 1 and append(Hkv=0) == 1 and append(cap=0) == 1
    assert append(hd=12) == 2 and append(hd=0) == 2
    assert append(kn=A + 8) == 3 and append(kc=4 * A + 4) == 3 and append(pos=3 * A + 2) == 3
    assert append(vc=4 * A) == 1                   # caches overlap
    assert append(B=0) == 0 and append(T=0, kn=0, vn=0, pos=0) == 0
    kc = fa.fa_prefill_kvcache
    args = (A, 2 * A, 3 * A, 4 * A, 1, 4, 2, 8)
    assert kc(*args, 9, 8, 128, 1, 0.1, 0, 0, 0, 0) == 1       # kv_len > kv_cap
    assert kc(*args, -1, 8, 128, 1, 0.1, 0, 0, 0, 0) == 1
    assert kc(*args, 8, 16, 100, 1, 0.1, 0, 0, 0, 0) == 2
    assert kc(*args, 8, 16, 128, 1, 0.1, 1, 5 * A + 16, 1 << 30, 0) == 3   # workspace not 256-aligned
    assert kc(A, 2 * A, 3 * A, 4 * A, 0, 4, 2, 8, 8, 16, 128, 1, 0.1, 0, 0, 0, 0) == 0  # B = 0


def test_paged_errors_without_a_device(fa):
    f = fa.fa_prefill_paged
    ok = dict(q=A, kp=8 * A, vp=16 * A, bt=24 * A, o=32 * A, B=1, Hq=4, Hkv=2, Sq=8, kv_len=300, hd=128, page=128,
              maxp=3, nb=4, causal=1, scale=0.1, bf16=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["kp"], a["vp"], a["bt"], a["o"], a["B"], a["Hq"], a["Hkv"], a["Sq"], a["kv_len"], a["hd"],
                 a["page"], a["maxp"], a["nb"], a["causal"], a["scale"], a["bf16"], 0)

    assert call(page=64) == 1 and call(page=200) == 1 and call(page=0) == 1   # not a multiple of 128
    assert call(maxp=2) == 1                      # 2 pages of 128 < 300 keys
    assert call(nb=0) == 1 and call(bt=0) == 1 and call(kv_len=-1) == 1
    assert call(bt=24 * A + 2) == 3 and call(hd=100) == 2 and call(hd=192) == 2  # paged: heads up to 128
    assert call(o=9 * A) == 1                     # o inside the K pool
    assert call(B=0) == 0


def test_ex_entry_point_errors_without_a_device(fa):
    f = fa.fa_prefill_ex
    args = (A, 2 * A, 3 * A, 4 * A)
    assert f(*args, 5 * A + 2, 1, 4, 2, 8, 8, 128, 1, 0.1, 0, 0, 0, 0) == 3       # misaligned lse
    assert f(*args, 4 * A, 1, 4, 2, 8, 8, 128, 1, 0.1, 0, 0, 0, 0) == 1           # lse inside o
    assert f(*args, 0, 1, 4, 2, 8, 8, 100, 1, 0.1, 0, 0, 0, 0) == 2
    assert f(*args, 0, 1, 4, 2, 8, 8, 256, 1, 0.1, 0, 6 * A, 1 << 30, 0) == 2     # split-KV: heads up to 128
    assert f(*args, 0, 1, 4, 2, 8, 8, 136, 1, 0.1, 0, 6 * A, 1 << 30, 0) == 2
    assert f(*args, 0, 0, 4, 2, 8, 8, 128, 1, 0.1, 0, 0, 0, 0) == 0               # B = 0


def test_force_path_values(fa):
    """fa_debug_force_path: 0 (library's choice) .. 3 (the CTA-pair kernel);
    anything else is rejected and leaves the setting alone.  Host-only."""
    lib = fa._lib.load()
    try:
        for path in (0, 1, 2, 3):
            assert lib.fa_debug_force_path(path) == 0
        for path in (-1, 4, 1000):
            assert lib.fa_debug_force_path(path) == 1  # FA_ERR_INVALID_ARG
        assert set(fa._lib.PATHS.values()) == {0, 1, 2, 3}
    finally:
        assert lib.fa_debug_force_path(0) == 0
