"""Synthetic workload definitions: layer shapes and input distributions.

Five layer shapes, from a tiny one the oracle finishes in well under a second
to a DeepSeek-V3-sized prefill.  Nothing here is arithmetic of the layer: it
only describes what the seeded input generator draws.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    n_experts: int
    n_sub: int
    I_sub: int
    k_max: int
    k_choices: Tuple[int, ...]          # uniform draw from these values
    k_per: str = "token"                # "token" or "request"
    tokens_per_request: int = 1
    score: str = "softmax"
    renorm: bool = False
    route_scale: float = 1.0
    router_std: Optional[float] = None  # None: N(0, 1/H) (variance 1/fan_in)
    bias: str = "none"                  # "none" | "normal" (N(0,1) per expert) | "zipf"
    zipf_s: float = 1.1
    I_shared: int = 0
    phase: str = "prefill"              # "prefill" or "decode" (what the bench reports)
    seed: int = 20261202
    native_m: int = 2                   # the original model's experts per token (proxy router)

    @property
    def E_r(self) -> int:
        return self.n_experts * self.n_sub

    @property
    def I(self) -> int:
        """Intermediate size of the monolithic expert the sub-experts slice."""
        return self.n_sub * self.I_sub

    def with_T(self, T: int) -> "Workload":
        base, _, tags = self.name.partition("@")
        tags = [t for t in tags.split("@") if t and not t.startswith("T")]
        return replace(self, T=T, name="@".join([base, *tags, f"T{T}"]))

    def with_experts(self, n: int) -> "Workload":
        base, _, tags = self.name.partition("@")
        tags = [t for t in tags.split("@") if t and not t.startswith("E")]
        return replace(self, n_experts=n, name="@".join([base, f"E{n}", *tags]))


# Tiny k-aware layer: 16 experts x 4 sub-experts of 128, k ~ U{1..8} per token.
TINY = Workload("tiny-h256-e16x4-t64", T=64, H=256, n_experts=16, n_sub=4, I_sub=128,
                k_max=8, k_choices=tuple(range(1, 9)), k_per="token", seed=20261202 + 0)

# Mixtral-8x7B-shaped decode step: 8 experts x 4 sub-experts of 3584, 64 one-token
# requests with k in {2,4,6,8}; per-expert logit bias ~ N(0,1).
MIXTRAL_DECODE = Workload("mixtral8x7b-decode-h4096-e8x4-t64", T=64, H=4096, n_experts=8,
                          n_sub=4, I_sub=3584, k_max=8, k_choices=(2, 4, 6, 8),
                          k_per="request", tokens_per_request=1, bias="normal",
                          phase="decode", seed=20261202 + 1)

# Qwen3-30B-A3B-shaped prefill: 128 experts (no split) of 768, 16 requests x 512
# tokens with k in {2,4,6,8} per request; router std 0.02 plus a Zipf(1.1) bias.
QWEN_PREFILL = Workload("qwen3-30b-a3b-prefill-h2048-e128-t8192", T=8192, H=2048,
                        n_experts=128, n_sub=1, I_sub=768, k_max=8, k_choices=(2, 4, 6, 8),
                        k_per="request", tokens_per_request=512, router_std=0.02,
                        bias="zipf", seed=20261202 + 2, native_m=8)

# Qwen3-30B-A3B-shaped decode sweep: 128 experts x 2 sub-experts of 384,
# T in {1, 8, 64, 256, 1024} one-token requests, k ~ U{4..16}.
QWEN_DECODE = Workload("qwen3-30b-a3b-decode-h2048-e128x2-t64", T=64, H=2048,
                       n_experts=128, n_sub=2, I_sub=384, k_max=16,
                       k_choices=tuple(range(4, 17)), k_per="token", phase="decode",
                       seed=20261202 + 3, native_m=8)
QWEN_DECODE_T = (1, 8, 64, 256, 1024)

# DeepSeek-V3-shaped prefill: 256 experts of 2048 plus one shared expert of 2048,
# 32 requests x 512 tokens with k in {4,6,8}; sigmoid scores renormalised.
DEEPSEEK_PREFILL = Workload("deepseek-v3-prefill-h7168-e256-shared-t16384", T=16384, H=7168,
                            n_experts=256, n_sub=1, I_sub=2048, k_max=8, k_choices=(4, 6, 8),
                            k_per="request", tokens_per_request=512, score="sigmoid",
                            renorm=True, I_shared=2048, seed=20261202 + 4, native_m=8)

ALL = {
    "tiny": TINY,
    "mixtral_decode": MIXTRAL_DECODE,
    "qwen_prefill": QWEN_PREFILL,
    "qwen_decode": QWEN_DECODE,
    "deepseek_prefill": DEEPSEEK_PREFILL,
}
