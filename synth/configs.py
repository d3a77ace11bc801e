"""The five workloads: shapes, value distributions and routing structure.

The shapes follow the two model families the Swiftlet pages name (the 35B
model routes each token to 8 of 256 experts, the 80B model to 10 of 512, each
MoE layer also holding one shared expert).  Hidden 2048, expert intermediate
512, group-64 MLX affine int4/int8 and the layer counts are the workload
definitions this build measures against.
"""
from __future__ import annotations

import dataclasses
import math

DEFAULT_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int
    bits: int = 4
    batches: tuple = (1,)
    steps: int = 256
    sigma: float = 0.02          # expert and shared-gate weights ~ N(0, sigma^2)
    router_sigma: float = 0.02   # router weights ~ N(0, router_sigma^2)
    zipf_s: float = 0.0          # 0 = no popularity bias
    pool_slots: int = 0          # 0 = all experts resident
    drift_swaps: int = 0         # adjacent-rank swaps per step and layer
    prefill_tokens: int = 0
    renorm: bool = True
    seed: int = DEFAULT_SEED

    @property
    def resident(self) -> bool:
        return self.pool_slots in (0, self.n_experts)

    def blob_bytes(self) -> int:
        """Packed bytes of one routed expert (nibble/byte codes + fp16 scale/bias)."""
        h, i, b = self.hidden, self.inter, self.bits
        q = 3 * h * i * b // 8
        sb = 3 * (h * i // 64) * 4
        return q + sb

    def blob_stride(self) -> int:
        return (self.blob_bytes() + 4095) // 4096 * 4096


CONFIGS = {
    # single layer, oracle in seconds; router seed chosen for a >= 1e-3 top-k gap
    "tiny": Workload("tiny", n_layers=1, hidden=256, n_experts=16, top_k=2, inter=128, shared_inter=128,
                     steps=1, renorm=False),
    # Qwen3.6-35B-A3B-shaped decode stack
    "35b": Workload("35b", n_layers=40, hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512),
    # Qwen3-Next-80B-A3B-shaped decode stack, logits ~ N(0,1) + Zipf(1.1) bias
    "80b": Workload("80b", n_layers=48, hidden=2048, n_experts=512, top_k=10, inter=512, shared_inter=512,
                    batches=(1, 8, 64), router_sigma=1.0 / math.sqrt(2048), zipf_s=1.1),
    # one 80B-shaped layer, 4096-token prefill
    "80b-prefill": Workload("80b-prefill", n_layers=1, hidden=2048, n_experts=512, top_k=10, inter=512,
                            shared_inter=512, router_sigma=1.0 / math.sqrt(2048), zipf_s=1.1,
                            prefill_tokens=4096, renorm=False),
    # streaming stress: 128 of 512 slots per layer, store in pinned host memory, drift
    "stress": Workload("stress", n_layers=48, hidden=2048, n_experts=512, top_k=10, inter=512,
                       shared_inter=512, router_sigma=1.0 / math.sqrt(2048), zipf_s=1.1, pool_slots=128,
                       drift_swaps=4, steps=1024),
}
