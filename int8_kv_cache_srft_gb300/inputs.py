"""Seeded synthetic inputs for the five KV-cache workloads.

This module only draws random tensors with the shapes, value distributions
and outlier structure of the workloads; it holds none of the codec's
arithmetic.  Tests feed the same tensors to the CUDA library and to the fp64
oracle, and ``bench.py`` times the library on them.  No model weights or
datasets are involved: the "Gemma-3-1B-shaped", "Qwen2.5-1.5B-shaped" and
"7B-like" caches borrow only the cache shapes of those models.

Cache tensors use the layout [n_outer][tokens][kv_heads][d] (fp16), where
n_outer is the layer index for the codec workloads and the batch index for
decode attention.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_outer: int          # layers (codec workloads) or batch (attention)
    tokens: int
    kv_heads: int
    d: int
    bits_k: int = 4
    bits_v: int = 4
    group: int = 16
    sign_seed: int = 1
    data_seed: int = 1
    lam: bool = False              # per-channel lambda ~ LogNormal(0, 0.5)
    outlier_kind: str = "none"     # "scale" | "student_t" | "none"
    outlier_channels: int = 0      # per (outer, kv head)
    outlier_factor: float = 1.0    # "scale": multiply the channel by this
    t_nu: int = 3                  # "student_t": degrees of freedom
    t_cap: int | None = None       # cache capacity in tokens (append workload)
    q_heads: int = 0               # attention workloads only
    extra: dict = field(default_factory=dict)

    @property
    def vectors_per_side(self) -> int:
        return self.n_outer * self.tokens * self.kv_heads

    def resized(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads.  Sign seed and data seed equal the workload number.
TINY = Workload("tiny round-trip [256 tokens x 2 kv heads x d=64], int4/int4 g16",
                n_outer=1, tokens=256, kv_heads=2, d=64, sign_seed=1, data_seed=1,
                outlier_kind="scale", outlier_channels=2, outlier_factor=20.0)
GEMMA = Workload("Gemma-3-1B-shaped cache [26 layers x 4096 tokens x 1 kv head x d=256], int4/int4 g16",
                 n_outer=26, tokens=4096, kv_heads=1, d=256, sign_seed=2, data_seed=2,
                 outlier_kind="student_t", outlier_channels=3, t_nu=3)
QWEN = Workload("Qwen2.5-1.5B-shaped outlier stress [28 layers x 32768 tokens x 2 kv heads x d=128], "
                "int4/int4 g16, per-channel lambda",
                n_outer=28, tokens=32768, kv_heads=2, d=128, sign_seed=3, data_seed=3, lam=True,
                outlier_kind="scale", outlier_channels=4, outlier_factor=50.0)
K8V4 = Workload("7B-like K8V4 append [32 layers x 8192 tokens x 8 kv heads x d=128], K int8 / V int4 g16",
                n_outer=32, tokens=8192, kv_heads=8, d=128, bits_k=8, bits_v=4, sign_seed=4, data_seed=4,
                t_cap=8192 + 1024)
DECODE = Workload("packed-cache decode attention [B=16, Hq=32, Hkv=8, d=128, T=131072], int4/int4 g16",
                  n_outer=16, tokens=131072, kv_heads=8, d=128, sign_seed=5, data_seed=5, q_heads=32)

WORKLOADS = {1: TINY, 2: GEMMA, 3: QWEN, 4: K8V4, 5: DECODE}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def kv_side(w: Workload, side: str, device="cpu", n_outer: int | None = None,
            tokens: int | None = None) -> torch.Tensor:
    """fp16 [n_outer][tokens][kv_heads][d] for side "k" or "v".

    Background N(0, 1); ``outlier_channels`` channels per (outer, kv head)
    either scaled by ``outlier_factor`` for every token or redrawn from a
    Student-t distribution with ``t_nu`` degrees of freedom.
    """
    n_outer = w.n_outer if n_outer is None else n_outer
    tokens = w.tokens if tokens is None else tokens
    seed = w.data_seed * 1000 + (1 if side == "k" else 2)
    g = _gen(seed, device)
    shape = (n_outer, tokens, w.kv_heads, w.d)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if w.outlier_kind != "none" and w.outlier_channels > 0:
        # the channel choice is drawn on the CPU so it does not depend on the device
        gc = _gen(seed + 7, "cpu")
        for o in range(n_outer):
            for h in range(w.kv_heads):
                ch = torch.randperm(w.d, generator=gc)[: w.outlier_channels].to(device)
                if w.outlier_kind == "scale":
                    x[o, :, h, ch] *= w.outlier_factor
                elif w.outlier_kind == "student_t":
                    zn = torch.randn((tokens, ch.numel()), generator=g, device=device)
                    chi = torch.randn((w.t_nu, tokens, ch.numel()), generator=g, device=device)
                    x[o, :, h, ch] = zn / torch.sqrt((chi * chi).sum(0) / w.t_nu)
                else:
                    raise ValueError(w.outlier_kind)
    return x.to(torch.float16)


def lam_table(w: Workload, side: str, device="cpu", n_outer: int | None = None) -> torch.Tensor | None:
    """fp32 [n_outer][kv_heads][d] per-channel lambda ~ LogNormal(0, 0.5), or None."""
    if not w.lam:
        return None
    n_outer = w.n_outer if n_outer is None else n_outer
    g = _gen(w.data_seed * 1000 + (11 if side == "k" else 12), device)
    return torch.exp(0.5 * torch.randn((n_outer, w.kv_heads, w.d), generator=g, device=device))


def query(w: Workload, device="cpu", batch: int | None = None) -> torch.Tensor:
    """fp16 [B][Hq][d] decode queries ~ N(0, 1)."""
    batch = w.n_outer if batch is None else batch
    g = _gen(w.data_seed * 1000 + 21, device)
    return torch.randn((batch, w.q_heads, w.d), generator=g, device=device).to(torch.float16)


def seq_lens(batch: int, t_cap: int, seed: int, device="cpu", ragged: bool = True) -> torch.Tensor:
    """int32 [B] sequence lengths: all t_cap, or a seeded ragged mix in [1, t_cap]."""
    if not ragged:
        return torch.full((batch,), t_cap, dtype=torch.int32, device=device)
    g = _gen(seed * 1000 + 31, "cpu")
    L = torch.randint(1, t_cap + 1, (batch,), generator=g, dtype=torch.int32)
    L[0] = t_cap
    return L.to(device)
