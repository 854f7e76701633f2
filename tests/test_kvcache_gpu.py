"""The K/V-cache path on a GB300, through the C ABI: the fused append
(fa_kv_append) bit for bit against the oracle's IEEE rounding and scatter, and
attention over a cache (fa_prefill_kvcache, both kernels) against the f64
oracle on the cache's valid rows -- with the rows past kv_len filled with NaN,
which must not reach the output (the pages' zero-staging rule, minfer "28 ·
r23 — f16-path whole-graph wall decomposition + FA_TKV occupancy raise",
section 3.2).  Tolerance for attention as in the parity tests:
|o - o_ref| <= tol (1 + |o_ref|), tol = 2e-3 (f16), 8e-3 (bf16)."""
import numpy as np
import pytest
import torch

import oracle
from causal_prefill_flash_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {False: 2e-3, True: 8e-3}


def _fa():
    import causal_prefill_flash_gb300 as fa
    return fa


def _f32_rows(shape, seed, specials=True):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32) * 4
    if specials:  # values that exercise rounding: overflow, subnormals, ties, NaN
        flat = x.view(-1)
        n = flat.numel()
        idx = torch.randperm(n, generator=g)[: min(n, 64)]
        vals = torch.tensor([7e4, -7e4, 65520.0, 6e-8, -3e-8, 2.0 ** -25, 1 + 2.0 ** -11, float("nan"),
                             3.4e38, 1e-40, -0.0, 2.0 ** -133], dtype=torch.float32)
        flat[idx] = vals[torch.arange(idx.numel()) % vals.numel()]
    return x


def _positions(B, T, cap, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.stack([torch.randperm(cap, generator=g)[:T] for _ in range(B)]).to(torch.int32)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("bf16", [False, True], ids=["f16", "bf16"])
@pytest.mark.parametrize("B,T,Hkv,hd,cap", [(1, 1, 1, 8, 1), (2, 37, 3, 64, 100), (3, 300, 8, 128, 1000),
                                            (2, 3000, 8, 128, 4096)])
def test_kv_append_matches_oracle_bit_for_bit(bf16, B, T, Hkv, hd, cap):
    fa = _fa()
    dt = torch.bfloat16 if bf16 else torch.float16
    k_new = _f32_rows((B, T, Hkv, hd), 100 + T)
    v_new = _f32_rows((B, T, Hkv, hd), 200 + T)
    pos = _positions(B, T, cap, 300 + T)
    sentinel_k = torch.full((B, cap, Hkv, hd), -7.0, dtype=dt)
    sentinel_v = torch.full((B, cap, Hkv, hd), 3.0, dtype=dt)
    kc, vc = sentinel_k.cuda(), sentinel_v.cuda()
    fa.kv_append(k_new.cuda(), v_new.cuda(), pos.cuda(), kc, vc)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    wk, wv = _bits(sentinel_k).copy(), _bits(sentinel_v).copy()
    assert oracle.kv_append(k_new.numpy(), v_new.numpy(), pos.numpy(), wk, wv, bf16=bf16) == 0
    gk, gv = _bits(kc), _bits(vc)
    e, m = (0x7F80, 0x007F) if bf16 else (0x7C00, 0x03FF)
    for got, want in ((gk, wk), (gv, wv)):
        nan_want = ((want & e) == e) & ((want & m) != 0)
        nan_got = ((got & e) == e) & ((got & m) != 0)
        assert np.array_equal(nan_got, nan_want)
        assert np.array_equal(got[~nan_want], want[~nan_want])


def test_kv_append_skips_and_reports_out_of_range_positions():
    fa = _fa()
    B, T, Hkv, hd, cap = 2, 6, 2, 64, 8
    k_new, v_new = _f32_rows((B, T, Hkv, hd), 1, False), _f32_rows((B, T, Hkv, hd), 2, False)
    pos = torch.tensor([[0, 1, 2, 3, 4, 5], [7, 6, 8, 5, 4, 3]], dtype=torch.int32)  # (1, 2) is out of range
    kc = torch.zeros((B, cap, Hkv, hd), dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    assert fa.debug_status_clear() == 0
    fa.kv_append(k_new.cuda(), v_new.cuda(), pos.cuda(), kc, vc)
    torch.cuda.synchronize()
    st = fa.debug_status()
    assert st & 0xFF == 32 and st >> 8 == 1 * T + 2, hex(st)
    assert fa.debug_status_clear() == 0
    wk = np.zeros((B, cap, Hkv, hd), dtype=np.uint16)
    wv = np.zeros_like(wk)
    assert oracle.kv_append(k_new.numpy(), v_new.numpy(), pos.numpy(), wk, wv, bf16=False) == 1
    assert np.array_equal(_bits(kc), wk) and np.array_equal(_bits(vc), wv)


@pytest.fixture(params=[False, True, "persistent"], ids=["oneshot", "splitkv", "persistent"])
def split(request):
    """The one-shot kernel; the split-KV path as the library routes it; and the
    split-KV schedule forced onto the persistent kernel."""
    if request.param != "persistent":
        yield request.param
        return
    request.getfixturevalue("force_persistent")
    yield True


@pytest.mark.parametrize("bf16", [False, True], ids=["f16", "bf16"])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,kv_len,cap,hd", [(1, 4, 2, 130, 700, 1024, 128), (2, 6, 2, 64, 300, 333, 64),
                                                      (1, 8, 8, 256, 256, 640, 128), (2, 4, 4, 1, 129, 200, 128)])
def test_attention_over_cache_ignores_rows_past_kv_len(bf16, B, Hq, Hkv, Sq, kv_len, cap, hd, split):
    fa = _fa()
    dt = torch.bfloat16 if bf16 else torch.float16
    w = W.Workload("case", B, Hq, Hkv, Sq, kv_len, hd, dtype="bf16" if bf16 else "f16", seed=kv_len + cap)
    q, k, v = W.make_inputs(w)
    kc = torch.full((B, cap, Hkv, hd), float("nan"), dtype=dt)
    vc = torch.full((B, cap, Hkv, hd), float("nan"), dtype=dt)
    kc[:, :kv_len], vc[:, :kv_len] = k, v
    out = torch.full_like(q, float("nan")).cuda()
    fa.attention_kvcache(q.cuda(), kc.cuda(), vc.cuda(), kv_len, causal=True, scale=w.scale, out=out, split=split)
    torch.cuda.synchronize()
    assert fa.debug_status() == 0
    got = out.cpu().double().numpy()
    want = oracle.attention(q, k, v, causal=True, scale=w.scale)
    err = np.abs(got - want) / (1 + np.abs(want))
    assert np.isfinite(got).all() and err.max() <= TOL[bf16], err.max()


def test_chunked_prefill_step_append_then_attend(split):
    """A chunked prefill over two chunks: each chunk's f32 K/V rows are appended
    at positions [kv_len, kv_len + T) of the cache, then the chunk's queries
    attend to rows [0, kv_len + T); the outputs match the oracle over the
    16-bit (rounded) K/V the cache holds."""
    fa = _fa()
    B, Hq, Hkv, hd, cap = 2, 8, 2, 128, 1024
    chunks = [300, 257]
    dt = torch.float16
    kc = torch.full((B, cap, Hkv, hd), float("nan"), dtype=dt, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    g = torch.Generator(device="cpu")
    g.manual_seed(5)
    k_all, v_all, kv_len = [], [], 0
    for T in chunks:
        k_new = torch.randn((B, T, Hkv, hd), generator=g, dtype=torch.float32)
        v_new = torch.randn((B, T, Hkv, hd), generator=g, dtype=torch.float32)
        q = torch.randn((B, T, Hq, hd), generator=g, dtype=torch.float32).to(dt)
        pos = (kv_len + torch.arange(T, dtype=torch.int32)).repeat(B, 1).contiguous()
        fa.kv_append(k_new.cuda(), v_new.cuda(), pos.cuda(), kc, vc)
        kv_len += T
        out = fa.attention_kvcache(q.cuda(), kc, vc, kv_len, causal=True, split=split)
        torch.cuda.synchronize()
        assert fa.debug_status() == 0
        # the oracle sees the K/V the append must have produced: the f32 rows rounded by the oracle
        for src, acc in ((k_new, k_all), (v_new, v_all)):
            bits = oracle.round16_bits(src.numpy(), bf16=False)
            acc.append(torch.from_numpy(bits.view(np.int16)).view(torch.float16))
        K, V = torch.cat(k_all, 1), torch.cat(v_all, 1)
        want = oracle.attention(q, K, V, causal=True, scale=1.0 / hd ** 0.5)
        got = out.cpu().double().numpy()
        err = np.abs(got - want) / (1 + np.abs(want))
        assert err.max() <= TOL[False], (T, err.max())
