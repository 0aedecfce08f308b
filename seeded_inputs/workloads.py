"""The synthetic FAVOR+ workloads: shapes, dtypes, feature family and seeds.

The pages measure on pixel, text and protein sequences ("Performer" paper note, *Evidence to
Read*), none of which is available here; these seeded Gaussian tensors stand in for them with
the shapes and value distributions below. Seeds: inputs 1234 + index, Omega 99 + index.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    m: int
    dtype: str            # "f32" or "bf16": storage type of Q, K, V, Omega and Y
    causal: bool
    kind: str = "exp"     # "exp" (FAVOR+ positive features) or "relu" (generalized ReLU)
    sigma: float = 1.0    # standard deviation of the raw Q, K, V entries
    chunk: int = 64       # causal chunk length
    relu_eps: float = 1e-3
    seed: int = 1234
    omega_seed: int = 99

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.n

    @property
    def heads(self) -> int:
        return self.B * self.H

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


_W = [
    # small fp32 non-causal case the oracle finishes in well under a second
    Workload("noncausal_f32_B1H1n256d64m128", 1, 1, 256, 64, 128, "f32", False),
    # the (1, 8, 1024, 64) shape of the linear-attention lesson's exercise, bf16 in / fp32 accumulate
    Workload("noncausal_bf16_B1H8n1024d64m256", 1, 8, 1024, 64, 256, "bf16", False),
    # causal, chunked prefix sums with 64-token chunks
    Workload("causal_bf16_B4H16n8192d64m256", 4, 16, 8192, 64, 256, "bf16", True, chunk=64),
    # long vision-token-shaped sequence, inputs N(0, 0.5^2)
    Workload("noncausal_bf16_B1H16n65536d128m256", 1, 16, 65536, 128, 256, "bf16", False, sigma=0.5),
    # causal generalized-ReLU features phi = ReLU(Omega x)/sqrt(m) + 1e-3
    Workload("causal_relu_bf16_B8H32n32768d64m512", 8, 32, 32768, 64, 512, "bf16", True, kind="relu"),
]
WORKLOADS = {}
for _i, _w in enumerate(_W):
    WORKLOADS[_w.name] = _w.with_(seed=1234 + _i, omega_seed=99 + _i)
WORKLOAD_ORDER = [w.name for w in _W]


def get_workload(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    raise KeyError(f"unknown workload {name!r}; known: {', '.join(WORKLOAD_ORDER)}")
