"""The workload shapes of the CSA2 attention step (sizes only, no arithmetic).

Sizes follow the model the pages describe: 64 query heads x 512, one shared
512-d latent per record serving as key and value, RoPE on the last 64 dims,
a 32-head x 128 lightning indexer, top-512 selection and a 128-token
sliding window ("DeepSeek V4 Inside", config table; "DeepSeek-V4.1-Flash
explained", sections 2, 3 and 7).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # sequences
    N: int                 # global records per sequence (decoder ratio 1: record j = position j)
    Bq: int                # query rows (B for decode, T for a prefill chunk)
    T: int = 0             # prefill chunk length; 0 = decode
    P0: int = 0            # prefill: position of the first new token
    q_pos_override: int = -1
    H: int = 64
    D: int = 512
    R: int = 64            # rotary dims (the last R of D)
    HI: int = 32           # indexer heads
    DI: int = 128          # indexer head dim
    K: int = 512           # top-K
    W: int = 128           # sliding window (rows attended, current token included)
    key_fmt: str = "bf16"  # indexer keys: "bf16" | "fp8" (E4M3 + fp32 row scale) | "mxfp4" (OCP MXFP4)
    lat_fmt: str = "bf16"  # latents: "bf16" | "fp4" (E2M1 + E4M3 group scale)
    lat_group: int = 32
    swa_fmt: str = "bf16"  # sliding-window rows: "bf16" | "fp8" (E4M3 + fp32 row scale)
    block_size: int = 64
    n_keep: int = 64
    n_reindex: int = 0     # hierarchical group: layers after the first that re-select from the pool
    n_reuse: int = 0       # layers after those that reuse the last selection
    hierarchical: bool = False
    n_hot_blocks: int = 0
    theta: float = 1e4

    @property
    def n_layers(self) -> int:
        return 1 + self.n_reindex + self.n_reuse

    @property
    def q_pos(self) -> int:
        """Decode: the query sits at position N and sees records 0..N-1."""
        return self.N if self.q_pos_override < 0 else self.q_pos_override

    def layer_mode(self, l: int) -> str:
        if l == 0:
            return "full_pool" if self.hierarchical else "full"
        if l <= self.n_reindex:
            return "reindex"
        return "reuse"


WORKLOADS = {
    "tiny_decode": Workload("tiny_decode", B=1, N=2048, Bq=1),
    "batched_decode": Workload("batched_decode", B=32, N=65536, Bq=32),
    "hierarchical": Workload("hierarchical", B=8, N=131072, Bq=8, hierarchical=True,
                             n_reindex=3, n_reuse=2, n_hot_blocks=96),
    "prefill_chunk": Workload("prefill_chunk", B=1, N=36864, Bq=4096, T=4096, P0=32768),
    "long_decode": Workload("long_decode", B=4, N=1048576, Bq=4, key_fmt="fp8",
                            lat_fmt="fp4", lat_group=32, swa_fmt="fp8"),
    # the pages' own indexer precision (OCP MXFP4 queries and keys) on the long-context shape
    "long_decode_mxfp4": Workload("long_decode_mxfp4", B=4, N=1048576, Bq=4, key_fmt="mxfp4",
                                  lat_fmt="fp4", lat_group=16, swa_fmt="fp8"),
}


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of ``wl`` with some sizes changed (for parity cases the oracle finishes quickly)."""
    if "T" in kw and "Bq" not in kw:
        kw["Bq"] = kw["T"]
    if "B" in kw and "Bq" not in kw and wl.T == 0:
        kw["Bq"] = kw["B"]
    return replace(wl, **kw)


@dataclass(frozen=True)
class ProjShape:
    """Sizes of the projections around attention: tokens, hidden size, query rank, heads,
    head size, output groups and output rank (the Flash config: hidden 4096, q rank 1024,
    64 heads of 512, 8 output groups; the output rank is not stated, 1024 is used)."""
    name: str
    tokens: int
    hidden: int = 4096
    q_rank: int = 1024
    heads: int = 64
    head_dim: int = 512
    groups: int = 8
    o_rank: int = 1024


PROJECTIONS = {
    "decode": ProjShape("decode", tokens=32),      # one decode step of the 32-sequence batch
    "prefill": ProjShape("prefill", tokens=4096),  # one 4096-token prefill chunk
}
