"""Workload geometries used by the tests and the benchmark.

Pure data: no attention arithmetic lives here. Shapes follow the VDN-Minimax-H3 window-attention article
(section 一: 102 latent frames, packed frame tokens plus text/audio global tokens, chunk-aligned windows with
radius r, "c1" = one chunk each side) and the MiniMax-H3 Ulysses pull request (Modifications, item 4: 56 heads).
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    T: int  # latent frames
    S: int  # spatial tokens per frame
    K: int  # frames per chunk
    r: int  # window radius in chunks
    G: int  # global tokens
    global_pos: int  # 0 = globals after the frame tokens, 1 = before them
    seed: int
    k_global_scale: float = 1.0  # multiplies the keys of the global rows before the bf16 cast

    @property
    def F(self) -> int:
        return self.T * self.S

    @property
    def L(self) -> int:
        return self.T * self.S + self.G

    @property
    def nc(self) -> int:
        return -(-self.T // self.K)

    @property
    def g0(self) -> int:
        return 0 if self.global_pos else self.T * self.S

    @property
    def f0(self) -> int:
        return self.G if self.global_pos else 0


TINY = Workload("tiny", B=1, H=2, D=64, T=6, S=16, K=2, r=1, G=8, global_pos=0, seed=1000)
MEDIUM = Workload("medium", B=1, H=8, D=128, T=24, S=256, K=4, r=1, G=256, global_pos=0, seed=1001)
H3 = Workload("h3", B=1, H=56, D=128, T=102, S=960, K=3, r=1, G=2048, global_pos=0, seed=1002,
              k_global_scale=2.0)
RAGGED = Workload("ragged", B=2, H=16, D=128, T=50, S=300, K=4, r=2, G=77, global_pos=1, seed=1003)


def sweep():
    """H3-shaped sweep: T in {34, 102}, K in {1, 3, 6}, r in {0, 1, 2}; H=56, D=128, S=960, G=2048 at the back."""
    pts = []
    i = 0
    for T in (34, 102):
        for K in (1, 3, 6):
            for r in (0, 1, 2):
                pts.append(Workload(f"sweep_T{T}_K{K}_r{r}", B=1, H=56, D=128, T=T, S=960, K=K, r=r, G=2048,
                                    global_pos=0, seed=2000 + i))
                i += 1
    return pts


# The H3-scale geometry with 8 of its 56 heads: per-head work is identical and q, k, v (205 MB each) are still
# larger than L2, so a profiler capture of it stands in for a full launch, scaled by 56 / 8.
H3_H8 = Workload("h3_h8", B=1, H=8, D=128, T=102, S=960, K=3, r=1, G=2048, global_pos=0, seed=1004,
                 k_global_scale=2.0)

ALL = {w.name: w for w in (TINY, MEDIUM, H3, RAGGED, H3_H8)}
