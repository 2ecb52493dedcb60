"""The named workloads of the chunked gated-delta-rule forward.

Each one is a single-GPU problem: (B, T, H, K, V, chunk), the gate kind, the io
dtype and whether the initial state is non-zero.  The 32k-token GDN problem is
the throughput workload; the 256-token fp32 problem is small enough for the
float64 oracle to check every output.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    chunk: int
    per_k_gate: bool
    io: str            # "f32" or "bf16"
    with_h0: bool

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.io == "f32" else torch.bfloat16

    @property
    def NT(self) -> int:
        return -(-self.T // self.chunk)     # a last, partial chunk counts

    @property
    def gate(self) -> str:
        return "kda" if self.per_k_gate else "gdn"

    def with_tokens(self, T: int) -> "Workload":
        """The same problem at another sequence length (for small profiling captures)."""
        if T <= 0:
            raise ValueError("T must be positive")
        name = self.name.replace(f"_t{self.T}_", f"_t{T}_")
        return replace(self, name=name, T=T)

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "T": self.T, "H": self.H,
                "K": self.K, "V": self.V, "chunk": self.chunk,
                "gate": "per_key_dim" if self.per_k_gate else "scalar",
                "io": self.io, "h0": "N(0,0.02)" if self.with_h0 else "zero"}


GDN_F32_T256 = Workload("gdn_f32_b1_t256_h2_d64_c64", 1, 256, 2, 64, 64, 64, False, "f32", False)
GDN_BF16_T2K = Workload("gdn_bf16_b4_t2048_h16_d128_c64", 4, 2048, 16, 128, 128, 64, False, "bf16", True)
GDN_BF16_C32 = Workload("gdn_bf16_b2_t4096_h8_d64_c32", 2, 4096, 8, 64, 64, 32, False, "bf16", False)
KDA_BF16_T8K = Workload("kda_bf16_b2_t8192_h16_d128_c64", 2, 8192, 16, 128, 128, 64, True, "bf16", False)
GDN_BF16_T32K = Workload("gdn_bf16_b1_t32768_h32_d128_c64", 1, 32768, 32, 128, 128, 64, False, "bf16", True)

ALL = [GDN_F32_T256, GDN_BF16_T2K, GDN_BF16_C32, KDA_BF16_T8K, GDN_BF16_T32K]

# Not one of the five problem configurations: the throughput workload's sequence with one eighth of
# its heads.  Its serial scan fills 16 of 152 SMs, the case the segment-parallel scan is for.
GDN_BF16_T32K_H4 = Workload("gdn_bf16_b1_t32768_h4_d128_c64", 1, 32768, 4, 128, 128, 64, False, "bf16", True)
EXTRA = [GDN_BF16_T32K_H4]

BY_NAME = {w.name: w for w in ALL + EXTRA}

# The long-context GDN problem is the one throughput is quoted on.
THROUGHPUT = GDN_BF16_T32K
