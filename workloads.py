"""Seeded synthetic inputs for the bf16 attention forward (no attention arithmetic here).

Both the oracle side and the CUDA side draw their inputs from this module and nothing
else; it holds no step of the method.  Shapes and value distributions follow the pages'
workloads: i.i.d. N(0, sigma^2) entries drawn in fp32 then rounded to bf16 (RTNE), in the
BSHD (B, S, H, d) or BHSD (B, H, S, d) layout, d = 128 (64 for one workload).  The named
workloads are a tiny self-attention, a square self-attention, a diffusion-style
cross-attention with a KV length that is not a tile multiple, a video-diffusion
self-attention (1536 hidden = 12 heads x 128), a long-KV stress case with large logits and
sparse non-finite entries, a decoder-style causal prefill whose K and V carry a quarter of
the query heads, and the square case at head dimension 64.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Skv: int
    d: int
    layout: str          # "bshd" or "bhsd"
    modes: tuple         # output rounding modes the workload is run under
    sigma: float = 1.0
    nonfinite_frac: float = 0.0   # fraction of K and V entries set to +inf/-inf/NaN
    seed: int = 0
    Hkv: int = 0                  # K/V heads; 0 means H (no grouping)
    causal: bool = False          # key j visible to query i iff j <= i + Skv - Sq

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H

    @property
    def visible_pairs(self) -> int:
        """Number of (query, key) pairs that take part, per (b, h)."""
        if not self.causal:
            return self.Sq * self.Skv
        off = self.Skv - self.Sq
        # row i sees min(max(i + off + 1, 0), Skv) keys
        return sum(min(max(i + off + 1, 0), self.Skv) for i in range(self.Sq))

    @property
    def flop(self) -> int:
        """4*d flops per visible (query, key) pair and head: the two matrix products (2*d
        each); 4*B*H*Sq*Skv*d without the causal mask."""
        return 4 * self.B * self.H * self.visible_pairs * self.d

    @property
    def min_bytes(self) -> int:
        """Q read and O written once, K and V (Hkv heads) read once, bf16."""
        return 2 * self.B * self.d * (2 * self.H * self.Sq + 2 * self.kv_heads * self.Skv)

    def describe(self) -> str:
        extra = (" Hkv=%d" % self.kv_heads if self.kv_heads != self.H else "") + \
                (" causal" if self.causal else "")
        return ("B=%d H=%d Sq=%d Skv=%d d=%d %s sigma=%g nonfinite=%g seed=%d%s"
                % (self.B, self.H, self.Sq, self.Skv, self.d, self.layout.upper(),
                   self.sigma, self.nonfinite_frac, self.seed, extra))


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 128, 128, "bshd", ("rtne",), seed=0),
    "square": Workload("square", 4, 16, 2048, 2048, 128, "bhsd", ("rtne", "rtna", "rtz"),
                       seed=1),
    "cross": Workload("cross", 2, 24, 4096, 300, 128, "bshd", ("rtne",), seed=2),
    "video": Workload("video", 1, 12, 32760, 32760, 128, "bshd", ("rtne", "rtz"), seed=3),
    "stress": Workload("stress", 1, 8, 128, 65536, 128, "bhsd", ("rtna",), sigma=4.0,
                       nonfinite_frac=1e-4, seed=4),
    # decoder-style prefill: causal mask with 4 query heads per K/V head
    "causal_gqa": Workload("causal_gqa", 2, 32, 8192, 8192, 128, "bshd", ("rtne",), seed=5,
                           Hkv=8, causal=True),
    # head dimension 64: the square self-attention's hidden size 2048 as 32 heads x 64
    "square_d64": Workload("square_d64", 4, 32, 2048, 2048, 64, "bhsd", ("rtne",), seed=6),
}


def shape(layout: str, B: int, H: int, S: int, d: int) -> tuple:
    return (B, S, H, d) if layout == "bshd" else (B, H, S, d)


def _randn_bf16(gen: torch.Generator, shp: tuple, sigma: float) -> torch.Tensor:
    x = torch.randn(shp, generator=gen, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(torch.bfloat16)


def _plant_nonfinite(gen: torch.Generator, t: torch.Tensor, frac: float) -> None:
    """Set round(frac * numel) seeded positions to +inf, -inf or NaN (chosen uniformly)."""
    n = int(round(frac * t.numel()))
    if n == 0:
        return
    flat = t.view(-1)
    pos = torch.randperm(t.numel(), generator=gen)[:n]
    kind = torch.randint(0, 3, (n,), generator=gen)
    vals = torch.tensor([float("inf"), float("-inf"), float("nan")], dtype=torch.bfloat16)
    flat[pos] = vals[kind]


def make_qkv(B: int, H: int, Sq: int, Skv: int, d: int = 128, layout: str = "bshd",
             seed: int = 0, sigma: float = 1.0, nonfinite_frac: float = 0.0, Hkv: int | None = None):
    """Draw Q, then K, then V (CPU bf16 tensors) from one seeded generator.  K and V carry
    ``Hkv`` heads (default H; fewer for grouped-query or multi-query attention)."""
    Hkv = H if Hkv is None else Hkv
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = _randn_bf16(gen, shape(layout, B, H, Sq, d), sigma)
    k = _randn_bf16(gen, shape(layout, B, Hkv, Skv, d), sigma)
    v = _randn_bf16(gen, shape(layout, B, Hkv, Skv, d), sigma)
    if nonfinite_frac > 0:
        _plant_nonfinite(gen, k, nonfinite_frac)
        _plant_nonfinite(gen, v, nonfinite_frac)
    return q, k, v


def make_workload(w: Workload):
    return make_qkv(w.B, w.H, w.Sq, w.Skv, w.d, w.layout, w.seed, w.sigma,
                    w.nonfinite_frac, Hkv=w.kv_heads)


def sample_rows(B: int, H: int, Sq: int, n: int, seed: int = 1234) -> torch.Tensor:
    """A seeded set of flat row indices (b*H + h)*Sq + i, always holding the first and the
    last row of every (b, h) so that ragged query tails are covered."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    total = B * H * Sq
    picks = torch.randint(0, total, (n,), generator=gen)
    edges = []
    for bh in range(B * H):
        edges += [bh * Sq, bh * Sq + Sq - 1]
    rows = torch.unique(torch.cat([picks, torch.tensor(edges, dtype=torch.int64)]))
    return rows
