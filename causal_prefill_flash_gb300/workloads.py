"""Seeded synthetic inputs for causal prefill attention.

This module holds no attention arithmetic: it only names the workloads (shapes,
dtypes, value distributions, seeds) and draws their Q, K, V.  Both the CUDA
path's tests/benchmark and the f64 oracle read inputs from here, so the two
sides always see bit-identical 16-bit tensors.

The workloads stand in for the prefill shapes of the 7B llama-style model the
minfer pages measure (hd = 128, 4 query heads per KV head in the GQA case,
2K / 2659 / 8192-token prompts, chunked prefill over a cached prefix); there is
no dataset and no weights: Q, K, V are i.i.d. normal draws from a CPU
``torch.Generator`` seeded with ``1234 + index``, drawn in float32, scaled by
the stated standard deviation and rounded to the workload's 16-bit type.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    hd: int
    causal: bool = True
    dtype: str = "f16"
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    seed: int = 1234
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.hd)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def visible_pairs(self) -> int:
        """Number of (query row, key) pairs the mask leaves visible, summed over B and Hq."""
        off = self.Skv - self.Sq
        if not self.causal:
            per_head = self.Sq * self.Skv
        else:
            per_head = 0
            for i in range(self.Sq):
                per_head += max(0, min(self.Skv, off + i + 1))
        return per_head * self.B * self.Hq

    def flops(self) -> int:
        """Algorithmic FLOPs: two contractions x 2 flops per multiply-add over visible pairs."""
        return 4 * self.hd * self.visible_pairs()

    def io_bytes(self) -> int:
        """Minimum HBM bytes: Q, K, V read once and O written once (16-bit elements)."""
        q = self.B * self.Sq * self.Hq * self.hd
        kv = self.B * self.Skv * self.Hkv * self.hd
        return 2 * (2 * q + 2 * kv)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The workload table, in the order the benchmark and the parity tests use it.
WORKLOADS = [
    Workload("single_head_s256", 1, 1, 1, 256, 256, 128, seed=1234,
             note="one head, Sq=Skv=256, f16 N(0,1)"),
    Workload("prefill7b_s2048", 1, 32, 32, 2048, 2048, 128, seed=1235,
             note="7B-shaped prefill, Sq=Skv=2048, f16 N(0,1)"),
    Workload("ragged_s2659_std3", 1, 32, 32, 2659, 2659, 128, q_std=3.0, k_std=3.0, seed=1236,
             note="non-tile-multiple prefill, Q,K ~ N(0,3^2) (std 3), V ~ N(0,1), f16"),
    Workload("gqa_s8192_bf16", 1, 32, 8, 8192, 8192, 128, dtype="bf16", seed=1237,
             note="GQA long prefill, 4 q heads per kv head, bf16 N(0,1)"),
    Workload("chunked_kv8192_hd128", 4, 32, 8, 512, 8192, 128, seed=1238,
             note="chunked prefill: 512 new rows over 7680 cached + 512 new keys, f16"),
    Workload("chunked_kv8192_hd64", 4, 32, 8, 512, 8192, 64, seed=1239,
             note="chunked prefill at hd=64, f16"),
    Workload("longctx_chunk128_kv32768", 1, 32, 8, 128, 32768, 128, seed=1240,
             note="a 128-row chunk over a 32640-token cached context: 16 query-tile pairs, "
                  "each 256 KV tiles long (an underfilled grid), f16"),
    Workload("encoder_s4096_noncausal", 2, 16, 16, 4096, 4096, 128, causal=False, dtype="bf16", seed=1241,
             note="encoder-style bidirectional attention (causal = 0): every row sees all 4096 keys, bf16"),
    Workload("gqa_s4096_hd256_bf16", 1, 16, 8, 4096, 4096, 256, dtype="bf16", seed=1242,
             note="head dimension 256 (16 query heads over 8 KV heads, the shape of 256-wide-head models), bf16"),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def get(name: str) -> Workload:
    return BY_NAME[name]


def make_inputs(w: Workload, device: str | torch.device = "cpu"):
    """Draw (q, k, v) for a workload: BSHD-contiguous tensors of the workload's 16-bit type."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    dt = w.torch_dtype
    q = (torch.randn((w.B, w.Sq, w.Hq, w.hd), generator=g, dtype=torch.float32) * w.q_std).to(dt)
    k = (torch.randn((w.B, w.Skv, w.Hkv, w.hd), generator=g, dtype=torch.float32) * w.k_std).to(dt)
    v = (torch.randn((w.B, w.Skv, w.Hkv, w.hd), generator=g, dtype=torch.float32) * w.v_std).to(dt)
    if str(device) != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def sample_rows(w: Workload, n: int, seed: int = 99):
    """A reproducible sample of output rows (b, hq, i) that always includes the
    first and last rows of the first and last heads plus random interior ones."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    fixed = {(0, 0, 0), (0, 0, w.Sq - 1), (w.B - 1, w.Hq - 1, 0), (w.B - 1, w.Hq - 1, w.Sq - 1)}
    rows = [r for r in sorted(fixed) if w.Sq > 0]
    while len(rows) < n:
        b = int(torch.randint(0, w.B, (1,), generator=g))
        h = int(torch.randint(0, w.Hq, (1,), generator=g))
        i = int(torch.randint(0, w.Sq, (1,), generator=g))
        rows.append((b, h, i))
    return torch.tensor(rows[:n], dtype=torch.int32)
