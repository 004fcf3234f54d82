"""The synthetic Qwen3-shaped workloads, as plain data.

Each workload fixes the cache geometry (batch, heads, head_dim, context,
group size), the L1 focal-set recipe (attention sinks + recent window +
seeded "reader-marked" tokens), the routing budget beta, the key
distribution and the storage type of K/V before encode.  Shapes follow the
Qwen3 family the Tamarin (HSQ) technical summary evaluates on (section 4,
Results: Qwen3 0.6B-14B, up to 32K context).  The heavy-tailed and low-rank
key laws follow the synthetic regimes of "Ablation, Statistical Inference,
and Validation for KV-Cache Compression" (technical summary, section 3,
regime-wise performance).
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # independent sequences
    Hq: int                # query heads
    Hkv: int               # KV heads
    T: int                 # context tokens already in the cache
    N: int                 # L2 group size
    beta: int              # groups fetched per KV head per step
    sinks: int             # attention-sink tokens at positions [0, sinks)
    recent: int            # recent window [T - recent, T)
    marked: int            # seeded reader-marked tokens drawn from [sinks, T - recent)
    storage: str           # "f32" or "bf16": type of K/V handed to encode
    key_law: str           # "lognormal" | "student_t" | "lowrank"
    steps: int             # decode steps in the workload
    layers: int = 1
    d: int = 128
    theta: float = 1.0e6
    needle: bool = False
    betas: Tuple[int, ...] = field(default_factory=tuple)  # beta sweep, if any
    seed_tag: int = 0      # distinguishes workloads in the seed tree

    @property
    def r(self) -> int:
        return self.Hq // self.Hkv

    @property
    def G(self) -> int:
        return -(-self.T // self.N)

    @property
    def l1_size(self) -> int:
        return self.sinks + self.recent + self.marked

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _frac(T: int, f: float) -> int:
    # "x% of the tokens" is read as floor(x * T).
    return int(f * T)


WORKLOADS = {
    # Tiny single layer: B1, 4 query / 2 KV heads, 1024 tokens, N=16,
    # L1 = 4 sinks + 64 recent + 32 random, beta = 8, fp32 inputs.
    "tiny_1k": Workload(
        name="tiny_1k", B=1, Hq=4, Hkv=2, T=1024, N=16, beta=8,
        sinks=4, recent=64, marked=32, storage="f32", key_law="lognormal",
        steps=16, seed_tag=0),
    # Qwen3-0.6B-shaped single layer: 16/8 heads, 4096 tokens, N=8,
    # L1 = 4 + 128 + 2% random, beta = 32, bf16 inputs.
    "qwen3_0p6b_4k": Workload(
        name="qwen3_0p6b_4k", B=1, Hq=16, Hkv=8, T=4096, N=8, beta=32,
        sinks=4, recent=128, marked=_frac(4096, 0.02), storage="bf16",
        key_law="lognormal", steps=256, seed_tag=1),
    # Qwen3-8B-shaped single layer at 32K: 32/8 heads, N=16 (2048 groups),
    # L1 = 4 + 256 + 1% marked, beta = 64, planted needle, bf16 inputs.
    "qwen3_8b_32k": Workload(
        name="qwen3_8b_32k", B=1, Hq=32, Hkv=8, T=32768, N=16, beta=64,
        sinks=4, recent=256, marked=_frac(32768, 0.01), storage="bf16",
        key_law="lognormal", steps=512, needle=True, seed_tag=2),
    # Qwen3-4B-shaped heavy-tailed batch decode: 16 sequences of 8192,
    # 32/8 heads, 36 layers, Student-t keys with 4 outlier channels x20.
    "qwen3_4b_b16_8k": Workload(
        name="qwen3_4b_b16_8k", B=16, Hq=32, Hkv=8, T=8192, N=8, beta=48,
        sinks=4, recent=128, marked=_frac(8192, 0.01), storage="bf16",
        key_law="student_t", steps=64, layers=36, seed_tag=3),
    # Qwen3-14B-shaped full step: 4 sequences of 32768, 40/8 heads,
    # 40 layers, low-rank keys, beta swept over {16, 64, 256}.
    "qwen3_14b_b4_32k": Workload(
        name="qwen3_14b_b4_32k", B=4, Hq=40, Hkv=8, T=32768, N=16, beta=64,
        sinks=4, recent=256, marked=_frac(32768, 0.01), storage="bf16",
        key_law="lowrank", steps=64, layers=40, betas=(16, 64, 256),
        seed_tag=4),
}


def get_workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.with_(**overrides) if overrides else w
