"""The MoE layer workloads, by model shape.

Each workload is one MoE layer: T tokens of hidden size d, E routed experts,
Top-K routing, SwiGLU experts of intermediate size F, optional capacity-factor
dropping per sub-sequence of S tokens, and (Qwen2-57B-A14B shape only) one
always-on shared SwiGLU expert of intermediate size Fs behind a sigmoid gate.

The four large shapes follow the models that the MoE Parallel Folding paper
benchmarks (study notes, "datasets, setup and metrics": Mixtral-8x22B,
Llama3-8x70B, Qwen2-57B-A14B, Mixtral-8x22B-G8T8, capacity factor 1 for the
token-drop runs). The tiny fp32 shape is a checking case.
"""
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens in the layer's batch (micro-batch x sequence, flattened)
    d: int            # hidden size
    E: int            # routed experts
    K: int            # Top-K
    F: int            # routed expert SwiGLU intermediate size
    dtype: str        # "f32" or "bf16": weights and activations
    drop: bool        # capacity-factor dropping (True) or dropless routing (False)
    cf: float = 1.0   # capacity factor (used when drop)
    S: int = 0        # sub-sequence length for dropping; 0 means S = T
    renorm: bool = True   # combine weights renormalised over the K selected experts
    Fs: int = 0       # shared expert intermediate size, 0 = no shared expert
    bias: bool = False    # per-expert router bias b_r ~ N(0, 1) (load skew)
    router_scale: float = 1.0  # router weight std multiplier (logits scale)
    backward: bool = False     # workload runs forward + backward
    seed: int = 0

    @property
    def subseq(self) -> int:
        return self.S if self.S > 0 else self.T

    @property
    def n_assign(self) -> int:
        return self.T * self.K

    def fwd_flops(self, n_kept: int) -> float:
        """Dense-contraction FLOPs of one forward: 6*N*d*F routed (+ 6*T*d*Fs shared)."""
        return 6.0 * n_kept * self.d * self.F + 6.0 * self.T * self.d * self.Fs

    def bwd_flops(self, n_kept: int) -> float:
        """Dense-contraction FLOPs of one backward: dgrad + wgrad = 12*N*d*F (+ shared)."""
        return 12.0 * n_kept * self.d * self.F + 12.0 * self.T * self.d * self.Fs


CONFIGS = {
    "tiny_f32": MoEConfig("tiny_f32", T=512, d=64, E=4, K=2, F=128, dtype="f32",
                          drop=False),
    "mixtral_8x22b": MoEConfig("mixtral_8x22b", T=8192, d=6144, E=8, K=2, F=16384,
                               dtype="bf16", drop=True, cf=1.0, S=4096),
    "qwen2_57b_a14b": MoEConfig("qwen2_57b_a14b", T=8192, d=3584, E=64, K=8, F=2560,
                                dtype="bf16", drop=False, Fs=20480, bias=True,
                                backward=True),
    "mixtral_8x22b_g8t8": MoEConfig("mixtral_8x22b_g8t8", T=16384, d=6144, E=64, K=8,
                                    F=2048, dtype="bf16", drop=True, cf=1.0, S=4096,
                                    backward=True),
    "llama3_8x70b": MoEConfig("llama3_8x70b", T=32768, d=8192, E=8, K=2, F=28672,
                              dtype="bf16", drop=False, router_scale=3.0,
                              backward=True),
}

# Reduced shapes with the same routing structure (E, K, mode, skew) that the CPU
# oracle finishes in seconds. Row counts per expert still span several 128-row
# tiles and leave ragged tails; d and F span several K-steps and N-tiles.
_SMALL = {
    "tiny_f32": dict(),
    "mixtral_8x22b": dict(T=1024, d=512, F=384, S=512),
    "qwen2_57b_a14b": dict(T=1024, d=512, F=256, Fs=512),
    "mixtral_8x22b_g8t8": dict(T=2048, d=512, F=256, S=512),
    "llama3_8x70b": dict(T=1024, d=768, F=384),
}


def get_config(name: str) -> MoEConfig:
    if name.endswith("@small"):
        return small_variant(name[: -len("@small")])
    return CONFIGS[name]


def small_variant(name: str) -> MoEConfig:
    base = CONFIGS[name]
    return replace(base, name=name + "@small", **_SMALL[name])
