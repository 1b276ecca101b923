"""The five synthetic workloads, by shape (no arithmetic here).

1. single expert, tiny: X [256, 512] N(0,1) with 1% outliers x20; W stored [256, 512] (K-major
   view of a 512x256 K x N matrix) N(0, 0.02); 4/6 on; requant of X^T and W^T with seed 0.
2. small grouped MoE forward: 8 experts, 4096 tokens, d_model 2048, SwiGLU width 1024, top-2.
3. Inkling-shaped MoE layer forward: 384 experts, top-8 of N(0,1) logits + per-expert N(0,1)
   bias, 16384 tokens, d_model 4096, SwiGLU width 2048, Student-t(3) activations.
4. backward requant stream: X [32768, 4096] Student-t(3); W [384, 2048, 4096] N(0, 0.02); Philox
   stochastic rounding with seeds 0..15.
5. full MoE layer step: workload-3 shapes, NVFP4 forward, MXFP8 backward GEMMs on requantised
   transposes, Hadamard(128) NVFP4 return path, FP32 master weights (SGD).
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class MoEShape:
    name: str
    tokens: int
    d_model: int
    d_ff: int
    experts: int
    top_k: int
    logit_bias: bool
    student_t: bool

    @property
    def rows(self) -> int:
        return self.tokens * self.top_k


SMALL_MOE = MoEShape("moe-small-e8-t4096-d2048-f1024-top2", 4096, 2048, 1024, 8, 2, False, False)
INKLING_MOE = MoEShape("inkling-moe-e384-t16384-d4096-f2048-top8", 16384, 4096, 2048, 384, 8, True,
                       True)

SINGLE_EXPERT = dict(name="single-expert-x256x512-w512x256", m=256, k=512, n=256)
REQUANT_STREAM = dict(name="requant-x32768x4096-w384x2048x4096", x_rows=32768, x_cols=4096,
                      w_experts=384, w_rows=2048, w_cols=4096, seeds=16)
