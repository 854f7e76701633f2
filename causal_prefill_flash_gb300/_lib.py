"""ctypes binding of libfa_prefill.so: argument marshalling only.

Every step of the attention computation runs in the library's CUDA kernel;
this module only turns tensors into pointers and sizes, passes the current
CUDA stream, and raises when the library returns an error.  There is no other
code path: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from ._build import LIB_PATH

_lock = threading.Lock()
_lib = None

FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_ALIGNMENT",
    4: "FA_ERR_SMEM", 5: "FA_ERR_LAUNCH", 6: "FA_ERR_DEVICE", 7: "FA_ERR_SCRATCH",
}

# (name, restype, argtypes) of every symbol include/fa_prefill.h declares
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIG = {
    "fa_prefill": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_prefill_bf16": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_prefill_ws": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, ctypes.c_size_t, _P]),
    "fa_prefill_ws_bf16": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, ctypes.c_size_t,
                                _P]),
    "fa_workspace_bytes": (ctypes.c_size_t, [_I]),
    "fa_split_kv_advised": (_I, [_I, _I, _I, _I, _I, _I]),
    "fa_split_kv_advised_hd": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_prefill_ex": (_I, [_P, _P, _P, _P, _P] + [_I] * 7 + [ctypes.c_float, _I, _P, ctypes.c_size_t, _P]),
    "fa_prefill_kvcache": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P,
                                ctypes.c_size_t, _P]),
    "fa_kv_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "fa_prefill_paged": (_I, [_P, _P, _P, _P, _P] + [_I] * 10 + [ctypes.c_float, _I, _P]),
    "fa_prefill_paged_ws": (_I, [_P, _P, _P, _P, _P] + [_I] * 10 + [ctypes.c_float, _I, _P, ctypes.c_size_t, _P]),
    "fa_prefill_ws_static": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_smem_bytes": (ctypes.c_uint, [_I]),
    "fa_debug_status": (_I, []),
    "fa_debug_status_clear": (_I, []),
    "fa_debug_set_watchdog_ns": (_I, [ctypes.c_ulonglong]),
    "fa_debug_force_path": (_I, [ctypes.c_int]),
    "fa_debug_schedule": (_I, [_I] * 7 + [_P, _P, _P, _I, _P]),
    "fa_debug_row_pairing": (_I, [_I] * 7),
}


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIG.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def smem_bytes(hd: int) -> int:
    return int(load().fa_smem_bytes(int(hd)))


def debug_status() -> int:
    return int(load().fa_debug_status())


def debug_status_clear() -> int:
    return int(load().fa_debug_status_clear())


def debug_set_watchdog_ns(ns: int) -> None:
    """Testing hook: the limit (ns) each pipeline wait of later launches may
    take before its CTA gives up and reports it (0 restores the 2 s default)."""
    load().fa_debug_set_watchdog_ns(int(ns))


PATHS = {"auto": 0, "oneshot": 1, "persistent": 2, "pair": 3}


def debug_force_path(path: str) -> None:
    """Testing hook: the kernel later calls run on -- "auto" (the library's
    choice), "oneshot" (the one-shot kernel, also for calls with a
    workspace), "persistent" (the persistent kernel: over whole units without
    a workspace, over every split-KV schedule with one) or "pair" (the
    CTA-pair kernel for calls it applies to: GQA groups of a multiple of 4
    query heads, heads 72 to 128 wide, contiguous K/V; the library's choice
    for the others)."""
    st = int(load().fa_debug_force_path(PATHS[path]))
    if st != FA_OK:
        raise FaError(st, "fa_debug_force_path")


def debug_schedule(B, Hq, Hkv, Sq, Skv, causal=True, sms=152):
    """The split-KV work split for a shape (host-only): a dict with the per-CTA
    start (pair, KV step) lists including the end entry, each pair's KV steps,
    the CTA count, whether every CTA runs one segment, the split pairs and the
    piece slots used."""
    n_max = 4096
    cp = (ctypes.c_int * 257)()
    cs = (ctypes.c_int * 257)()
    ps = (ctypes.c_int * n_max)()
    out = (ctypes.c_int * 4)()
    nu = int(load().fa_debug_schedule(int(B), int(Hq), int(Hkv), int(Sq), int(Skv), int(bool(causal)), int(sms),
                                      ctypes.addressof(cp), ctypes.addressof(cs), ctypes.addressof(ps), n_max,
                                      ctypes.addressof(out)))
    if nu < 0:
        raise FaError(-nu, "fa_debug_schedule")
    G = out[0]
    return {"pairs": nu, "ctas": G, "one_segment": bool(out[1]), "split_pairs": out[2], "slots": out[3],
            "cta_pair": list(cp[: G + 1]), "cta_step": list(cs[: G + 1]), "pair_steps": list(ps[:nu])}


def debug_row_pairing(B, Hq, Hkv, Sq, Skv, causal=True, sms=152) -> bool:
    """Whether the one-shot grid leaves query tile 0 without a partner (True)
    or the last tile (False, also when no tile goes alone) for a shape on a
    GPU of ``sms`` SMs (host-only)."""
    st = int(load().fa_debug_row_pairing(int(B), int(Hq), int(Hkv), int(Sq), int(Skv), int(bool(causal)), int(sms)))
    if st < 0:
        raise FaError(-st, "fa_debug_row_pairing")
    return bool(st)


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(getattr(stream, "cuda_stream", stream))


def fa_prefill(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, stream=None) -> int:
    """f16 entry point: same arguments as the C function (tensors or raw device
    pointers for q/k/v/o; ``stream`` None = torch's current stream). Returns the status."""
    return int(load().fa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), int(B), int(Hq), int(Hkv), int(Sq),
                                 int(Skv), int(hd), int(causal), float(scale), _stream(stream)))


def fa_prefill_bf16(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, stream=None) -> int:
    """bf16 entry point: same arguments as the C function. Returns the status."""
    return int(load().fa_prefill_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), int(B), int(Hq), int(Hkv), int(Sq),
                                      int(Skv), int(hd), int(causal), float(scale), _stream(stream)))


def fa_prefill_ws(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, workspace, workspace_bytes,
                  stream=None) -> int:
    """Stream-K entry point (f16): the C function's arguments. Returns the status."""
    return int(load().fa_prefill_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), int(B), int(Hq), int(Hkv), int(Sq),
                                    int(Skv), int(hd), int(causal), float(scale), _ptr(workspace),
                                    int(workspace_bytes), _stream(stream)))


def fa_prefill_ws_bf16(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, workspace, workspace_bytes,
                       stream=None) -> int:
    """Stream-K entry point (bf16): the C function's arguments. Returns the status."""
    return int(load().fa_prefill_ws_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), int(B), int(Hq), int(Hkv),
                                         int(Sq), int(Skv), int(hd), int(causal), float(scale), _ptr(workspace),
                                         int(workspace_bytes), _stream(stream)))


def fa_prefill_ws_static(q, k, v, o, B, Hq, Hkv, Sq, Skv, hd, causal, scale, bf16, stream=None) -> int:
    """Split-KV entry point with the library's static scratch: the C function's
    arguments (``bf16`` 0 for f16, 1 for bfloat16).  Allocates nothing: for
    callers that cannot allocate device memory at call time.  Returns the status."""
    return int(load().fa_prefill_ws_static(_ptr(q), _ptr(k), _ptr(v), _ptr(o), int(B), int(Hq), int(Hkv),
                                           int(Sq), int(Skv), int(hd), int(causal), float(scale), int(bf16),
                                           _stream(stream)))


def fa_prefill_kvcache(q, k_cache, v_cache, o, B, Hq, Hkv, Sq, kv_len, kv_cap, hd, causal, scale, bf16,
                       workspace=None, workspace_bytes=0, stream=None) -> int:
    """Attention over a K/V cache: the C function's arguments. Returns the status."""
    return int(load().fa_prefill_kvcache(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), int(B), int(Hq),
                                         int(Hkv), int(Sq), int(kv_len), int(kv_cap), int(hd), int(causal),
                                         float(scale), int(bf16), _ptr(workspace), int(workspace_bytes),
                                         _stream(stream)))


def fa_prefill_paged(q, k_pool, v_pool, block_table, o, B, Hq, Hkv, Sq, kv_len, hd, page_size, max_pages,
                     num_blocks, causal, scale, bf16, stream=None) -> int:
    """Attention over a paged K/V pool: the C function's arguments. Returns the status."""
    return int(load().fa_prefill_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(o), int(B),
                                       int(Hq), int(Hkv), int(Sq), int(kv_len), int(hd), int(page_size),
                                       int(max_pages), int(num_blocks), int(causal), float(scale), int(bf16),
                                       _stream(stream)))


def fa_prefill_paged_ws(q, k_pool, v_pool, block_table, o, B, Hq, Hkv, Sq, kv_len, hd, page_size, max_pages,
                        num_blocks, causal, scale, bf16, workspace, workspace_bytes, stream=None) -> int:
    """Split-KV attention over a paged K/V pool: the C function's arguments. Returns the status."""
    return int(load().fa_prefill_paged_ws(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(o),
                                          int(B), int(Hq), int(Hkv), int(Sq), int(kv_len), int(hd),
                                          int(page_size), int(max_pages), int(num_blocks), int(causal),
                                          float(scale), int(bf16), _ptr(workspace), int(workspace_bytes),
                                          _stream(stream)))


def attention_paged(q, k_pool, v_pool, block_table, kv_len: int, causal: bool = True,
                    scale: float | None = None, out=None, stream=None, split: bool | None = None):
    """O = softmax(scale Q K^T + causal mask) V with K, V read from pools
    [num_blocks, page_size, Hkv, hd] through block_table [B, max_pages]
    (int32): key j of sequence b is k_pool[block_table[b, j // page_size],
    j % page_size].  page_size must be a multiple of 128.  ``split`` as in
    ``attention`` (split-KV for heads up to 128 wide).  Raises FaError."""
    import torch
    if q.dim() != 4 or k_pool.dim() != 4 or v_pool.shape != k_pool.shape or block_table.dim() != 2:
        raise ValueError("q [B, Sq, Hq, hd], pools [num_blocks, page_size, Hkv, hd], table [B, max_pages]")
    if not (q.dtype == k_pool.dtype == v_pool.dtype) or q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("q and the pools must all be float16 or all bfloat16")
    if block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32")
    for t in (q, k_pool, v_pool, block_table):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    B, Sq, Hq, hd = q.shape
    num_blocks, page_size, Hkv, hdk = k_pool.shape
    if hdk != hd or block_table.shape[0] != B:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor like q")
    if split is None:
        split = hd <= 128 and split_kv_advised(B, Hq, Hkv, Sq, kv_len, causal, hd)
    if split:
        ws = workspace_for(q.device, hd, stream)
        st = fa_prefill_paged_ws(q, k_pool, v_pool, block_table, out, B, Hq, Hkv, Sq, kv_len, hd, page_size,
                                 block_table.shape[1], num_blocks, int(bool(causal)), scale,
                                 int(q.dtype == torch.bfloat16), ws, ws.numel(), stream)
    else:
        st = fa_prefill_paged(q, k_pool, v_pool, block_table, out, B, Hq, Hkv, Sq, kv_len, hd, page_size,
                              block_table.shape[1], num_blocks, int(bool(causal)), scale,
                              int(q.dtype == torch.bfloat16), stream)
    if st != FA_OK:
        raise FaError(st, "fa_prefill_paged_ws" if split else "fa_prefill_paged")
    return out


def fa_kv_append(k_new, v_new, positions, k_cache, v_cache, B, T, Hkv, hd, kv_cap, bf16, stream=None) -> int:
    """K/V-cache append: the C function's arguments. Returns the status."""
    return int(load().fa_kv_append(_ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(k_cache), _ptr(v_cache),
                                   int(B), int(T), int(Hkv), int(hd), int(kv_cap), int(bf16), _stream(stream)))


def kv_append(k_new, v_new, positions, k_cache, v_cache, stream=None):
    """Write the f32 rows k_new, v_new [B, T, Hkv, hd] into the 16-bit caches
    [B, kv_cap, Hkv, hd] at rows positions [B, T] (int32), rounded to the
    caches' dtype.  All CUDA tensors, contiguous.  Raises FaError on error."""
    import torch
    if k_new.dtype != torch.float32 or v_new.dtype != torch.float32:
        raise ValueError("k_new and v_new must be float32")
    if k_cache.dtype != v_cache.dtype or k_cache.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("caches must both be float16 or both bfloat16")
    if positions.dtype != torch.int32:
        raise ValueError("positions must be int32")
    for t in (k_new, v_new, positions, k_cache, v_cache):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    B, T, Hkv, hd = k_new.shape
    if v_new.shape != k_new.shape or positions.shape != (B, T) or k_cache.shape != v_cache.shape \
            or k_cache.dim() != 4 or k_cache.shape[0] != B or k_cache.shape[2:] != (Hkv, hd):
        raise ValueError("shape mismatch")
    st = fa_kv_append(k_new, v_new, positions, k_cache, v_cache, B, T, Hkv, hd, k_cache.shape[1],
                      int(k_cache.dtype == torch.bfloat16), stream)
    if st != FA_OK:
        raise FaError(st, "fa_kv_append")


def attention_kvcache(q, k_cache, v_cache, kv_len: int, causal: bool = True, scale: float | None = None,
                      out=None, stream=None, split: bool | None = None):
    """O = softmax(scale Q K^T + causal mask) V over the first kv_len rows of
    the caches [B, kv_cap, Hkv, hd] (the query rows are the last Sq of those
    kv_len positions).  ``split`` as in ``attention``.  Raises FaError."""
    import torch
    if q.dim() != 4 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("q must be [B, Sq, Hq, hd] and the caches [B, kv_cap, Hkv, hd]")
    if not (q.dtype == k_cache.dtype == v_cache.dtype) or q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("q and the caches must all be float16 or all bfloat16")
    for t in (q, k_cache, v_cache):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("q and the caches must be contiguous CUDA tensors")
    B, Sq, Hq, hd = q.shape
    Bk, kv_cap, Hkv, hdk = k_cache.shape
    if Bk != B or hdk != hd:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor like q")
    if split is None:
        split = hd <= 128 and split_kv_advised(B, Hq, Hkv, Sq, kv_len, causal, hd)
    ws = workspace_for(q.device, hd, stream) if split else None
    st = fa_prefill_kvcache(q, k_cache, v_cache, out, B, Hq, Hkv, Sq, kv_len, kv_cap, hd, int(bool(causal)),
                            scale, int(q.dtype == torch.bfloat16), ws, ws.numel() if ws is not None else 0, stream)
    if st != FA_OK:
        raise FaError(st, "fa_prefill_kvcache")
    return out


def fa_prefill_ex(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, hd, causal, scale, bf16, workspace=None,
                  workspace_bytes=0, stream=None) -> int:
    """Any hd, either kernel, optional log-sum-exp: the C function's arguments. Returns the status."""
    return int(load().fa_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv),
                                    int(Sq), int(Skv), int(hd), int(causal), float(scale), int(bf16),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream)))


def split_kv_advised(B, Hq, Hkv, Sq, Skv, causal=True, hd=None) -> bool:
    """The library's advice for this shape on the current device: True when the
    split-KV path is expected to beat the one-shot kernel.  With ``hd`` the
    head-width-aware rule (fa_split_kv_advised_hd) is used."""
    if hd is None:
        st = int(load().fa_split_kv_advised(int(B), int(Hq), int(Hkv), int(Sq), int(Skv), int(bool(causal))))
    else:
        st = int(load().fa_split_kv_advised_hd(int(B), int(Hq), int(Hkv), int(Sq), int(Skv), int(hd),
                                               int(bool(causal))))
    if st < 0:
        raise FaError(-st, "fa_split_kv_advised")
    return st == 1


def workspace_bytes(hd: int) -> int:
    return int(load().fa_workspace_bytes(int(hd)))


_workspaces = {}


def workspace_for(device, hd: int, stream=None):
    """A workspace for the stream-K path, one per (device, stream, hd), allocated
    once by torch and reused (calls on one stream never overlap; the kernels
    read only what the same call wrote, so it needs no initialisation)."""
    import torch
    key = (str(device), int(_stream(stream)) if stream is not None else None, int(hd))
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.empty(workspace_bytes(hd), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def attention(q, k, v, causal: bool = True, scale: float | None = None, out=None, stream=None,
              split: bool | None = None, return_lse: bool = False):
    """O = softmax(scale Q K^T + causal mask) V for BSHD CUDA tensors.

    q: [B, Sq, Hq, hd], k/v: [B, Skv, Hkv, hd], all float16 or all bfloat16,
    contiguous, on the current CUDA device.  Returns O with q's shape and dtype
    (written into ``out`` when given).  ``split=True`` uses the load-balanced
    stream-K (split-KV) kernel with a cached workspace, ``split=False`` the
    one-shot kernel, ``split=None`` whichever the library advises for the
    shape (``split_kv_advised``).  ``return_lse=True`` also returns the
    per-row log-sum-exp of the scaled scores, float32 [B, Hq, Sq] (-inf for a
    row that sees no key).  Raises FaError on any library error.
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("q, k, v must all be float16 or all bfloat16")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, Sq, Hq, hd] and k, v [B, Skv, Hkv, hd]")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous (BSHD)")
    B, Sq, Hq, hd = q.shape
    Bk, Skv, Hkv, hdk = k.shape
    if Bk != B or hdk != hd:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor like q")
    if split is None:  # split-KV exists for heads up to 128 wide
        split = hd <= 128 and split_kv_advised(B, Hq, Hkv, Sq, Skv, causal, hd)
    if return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
        ws = workspace_for(q.device, hd, stream) if split else None
        st = fa_prefill_ex(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, hd, int(bool(causal)), scale,
                           int(q.dtype == torch.bfloat16), ws, ws.numel() if ws is not None else 0, stream)
        if st != FA_OK:
            raise FaError(st, "fa_prefill_ex")
        return out, lse
    if split:
        fn = fa_prefill_ws_bf16 if q.dtype == torch.bfloat16 else fa_prefill_ws
        ws = workspace_for(q.device, hd, stream)
        st = fn(q, k, v, out, B, Hq, Hkv, Sq, Skv, hd, int(bool(causal)), scale, ws, ws.numel(), stream)
    else:
        fn = fa_prefill_bf16 if q.dtype == torch.bfloat16 else fa_prefill
        st = fn(q, k, v, out, B, Hq, Hkv, Sq, Skv, hd, int(bool(causal)), scale, stream)
    if st != FA_OK:
        raise FaError(st, fn.__name__)
    return out
