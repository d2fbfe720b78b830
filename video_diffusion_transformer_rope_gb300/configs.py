"""The five Wan-shaped attention workloads this library is measured and checked on.

Shapes follow the Wan2.1 latent grids named on the vidax page ("vidax: A Unified JAX
Framework for Video Generative Models on Accelerator Meshes", §4 "Experimental setup" and
App. B: batch 1 with classifier-free guidance, i.e. an internal batch of 2; 480p and native
720p Wan2.1 1.3B / 14B).  Token index n = t*Hg*Wg + h*Wg + w.
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int          # attention heads
    d: int          # head_dim
    T: int          # latent frames
    Hg: int         # latent grid height
    Wg: int         # latent grid width
    dtype: str      # "f32" or "bf16": element type of q, k, v and out
    sections: tuple  # rotary dims per axis (t, h, w), each even, summing to d
    theta: float = 10000.0
    seed: int = 0
    stress: bool = False   # outlier channels/tokens (large-logit softmax stress)
    # QK operand precision the workload is run with: "fp16" (default) or "split" (hi + lo fp16
    # parts, for logits in the hundreds, where 11 significant bits leave lse errors of ~0.1)
    qk: str = "fp16"

    @property
    def N(self) -> int:
        return self.T * self.Hg * self.Wg

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    @property
    def flops(self) -> float:
        """Algorithmic work of one call: QK^T plus PV, 2 FLOP per multiply-add each."""
        return 4.0 * self.B * self.H * float(self.N) ** 2 * self.d

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} H={self.H} d={self.d} grid {self.T}x{self.Hg}x{self.Wg} "
                f"(N={self.N}) {self.dtype} sections {self.sections[0]}/{self.sections[1]}/"
                f"{self.sections[2]} theta={self.theta:g}")


TINY_F32 = Workload("tiny_f32", B=1, H=4, d=64, T=3, Hg=8, Wg=8, dtype="f32",
                    sections=(24, 20, 20), seed=0)
WAN13B_480P = Workload("wan1.3b_480p", B=2, H=12, d=128, T=21, Hg=30, Wg=52, dtype="bf16",
                       sections=(44, 42, 42), seed=1)
WAN14B_480P = Workload("wan14b_480p", B=2, H=40, d=128, T=21, Hg=30, Wg=52, dtype="bf16",
                       sections=(44, 42, 42), seed=2)
WAN14B_720P = Workload("wan14b_720p", B=2, H=40, d=128, T=21, Hg=45, Wg=80, dtype="bf16",
                       sections=(44, 42, 42), seed=3)
LONG_STRESS = Workload("long_clip_stress", B=1, H=40, d=128, T=31, Hg=45, Wg=80, dtype="bf16",
                       sections=(44, 42, 42), seed=4, stress=True, qk="split")

ALL = (TINY_F32, WAN13B_480P, WAN14B_480P, WAN14B_720P, LONG_STRESS)
BY_NAME = {w.name: w for w in ALL}
