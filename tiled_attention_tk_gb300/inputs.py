"""Seeded synthetic attention inputs.

This module only draws random numbers; it holds none of the attention
arithmetic.  Tests, the smoke check and the benchmark use it to feed the
same bf16 tensors to the CUDA library and to the CPU oracle.

Recipe: ``torch.Generator('cpu').manual_seed(seed)``; values are drawn in
fp32 and rounded to bf16 (round to nearest even) with ``.to(torch.bfloat16)``.
Q, K and V of workload ``c`` take seeds ``1000*c + 0``, ``+1`` and ``+2``.
Layout: contiguous ``[B, H, N, D]``.

The workloads below are the attention-forward shapes this library is
measured on (the sixth: queries against a longer key sequence); the pages that describe the method print no shapes of their own
besides head dims 64 and 128 (the "ThunderKittens" attention kernel on
10100.com/article/71410160, section "writing a kernel with TK",
attn_fwd_layout).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    index: int
    B: int
    H: int
    N: int
    D: int
    causal: bool
    dist: str  # "normal": Q,K,V ~ N(0,1); "wide": Q,K ~ N(0,3^2), V ~ U(-1,1)
    kv_len: int | None = None  # key/value rows when they differ from the N query rows

    @property
    def Nkv(self) -> int:
        return self.N if self.kv_len is None else self.kv_len

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def name(self) -> str:
        kv = f"Nkv{self.Nkv}" if self.Nkv != self.N else ""
        return (f"B{self.B}H{self.H}N{self.N}{kv}D{self.D}"
                f"{'-causal' if self.causal else ''}{'-wide' if self.dist == 'wide' else ''}")

    @property
    def flops(self) -> float:
        """Algorithmic flops of the two contractions: 4*B*H*N*Nkv*D, with the
        causal mask 4*B*H*D*(N*(Nkv-N) + N^2/2) (masked products are not
        counted; for Nkv = N that is half of the unmasked count)."""
        if self.causal:
            return 4.0 * self.B * self.H * self.D * (self.N * (self.Nkv - self.N) + self.N * self.N / 2.0)
        return 4.0 * self.B * self.H * self.N * self.Nkv * self.D

    def describe(self) -> dict:
        d = {"workload": self.name, "B": self.B, "H": self.H, "N": self.N}
        if self.Nkv != self.N:
            d["Nkv"] = self.Nkv
        return dict(d, **{"D": self.D, "causal": self.causal,
                "dist": ("Q,K,V~N(0,1)" if self.dist == "normal"
                         else "Q,K~N(0,3^2), V~U(-1,1)"),
                "scale": f"1/sqrt({self.D})"})


WORKLOADS = {
    1: Workload(1, 1, 1, 128, 64, False, "normal"),
    2: Workload(2, 4, 16, 2048, 64, False, "normal"),
    3: Workload(3, 4, 16, 4096, 128, True, "normal"),
    4: Workload(4, 16, 32, 1024, 128, False, "wide"),
    5: Workload(5, 1, 32, 16384, 128, True, "normal"),
    # 2048 new queries at the end of a 16384-key sequence (attention
    # inference over a cache)
    6: Workload(6, 1, 32, 2048, 128, True, "normal", kv_len=16384),
}


def _draw(shape, seed: int, kind: str, std: float = 1.0) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    if kind == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
    elif kind == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32).mul_(2.0).sub_(1.0)
    else:
        raise ValueError(kind)
    return x.to(torch.bfloat16)


def make_qkv(B: int, H: int, N: int, D: int, seed_base: int, dist: str = "normal"):
    """Q, K, V as contiguous bf16 CPU tensors of shape [B,H,N,D]."""
    shape = (B, H, N, D)
    if dist == "normal":
        return (_draw(shape, seed_base + 0, "normal"),
                _draw(shape, seed_base + 1, "normal"),
                _draw(shape, seed_base + 2, "normal"))
    if dist == "wide":
        return (_draw(shape, seed_base + 0, "normal", 3.0),
                _draw(shape, seed_base + 1, "normal", 3.0),
                _draw(shape, seed_base + 2, "uniform"))
    raise ValueError(dist)


def make_qkv_rect(B: int, H: int, Nq: int, Nkv: int, D: int, seed_base: int, dist: str = "normal"):
    """Q [B,H,Nq,D] and K, V [B,H,Nkv,D], contiguous bf16 CPU tensors, drawn
    like make_qkv (same seeds and distributions)."""
    if dist == "normal":
        return (_draw((B, H, Nq, D), seed_base + 0, "normal"),
                _draw((B, H, Nkv, D), seed_base + 1, "normal"),
                _draw((B, H, Nkv, D), seed_base + 2, "normal"))
    if dist == "wide":
        return (_draw((B, H, Nq, D), seed_base + 0, "normal", 3.0),
                _draw((B, H, Nkv, D), seed_base + 1, "normal", 3.0),
                _draw((B, H, Nkv, D), seed_base + 2, "uniform"))
    raise ValueError(dist)


def workload_inputs(w: Workload):
    """The seeded inputs of one of the named workloads."""
    if w.Nkv != w.N:
        return make_qkv_rect(w.B, w.H, w.N, w.Nkv, w.D, 1000 * w.index, w.dist)
    return make_qkv(w.B, w.H, w.N, w.D, 1000 * w.index, w.dist)


def sample_heads(w: Workload, count: int, seed: int = 7):
    """A seeded sample of ``count`` distinct (b, h) pairs that always contains
    the first and the last head."""
    total = w.B * w.H
    if count >= total:
        return [(i // w.H, i % w.H) for i in range(total)]
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + w.index)
    chosen = {0, total - 1}
    perm = torch.randperm(total, generator=g).tolist()
    for i in perm:
        if len(chosen) >= count:
            break
        chosen.add(i)
    return [(i // w.H, i % w.H) for i in sorted(chosen)]


def sample_rows(N: int, count: int, seed: int = 11, tile: int = 128):
    """Seeded query rows of one head: the first and last rows, rows on both
    sides of every few 128-row tile boundaries, and random rows."""
    rows = {0, 1, N - 1, N - 2}
    for b in range(tile, N, tile * max(1, (N // tile) // 8)):
        rows.update({b - 1, b, b + 1})
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + N)
    extra = torch.randint(0, N, (count,), generator=g).tolist()
    rows.update(extra)
    return sorted(r for r in rows if 0 <= r < N)
