"""Workload shapes of the sparse offloaded-KV decode step.

Each workload is one decode step of landmark-based sparse attention over a KV
cache kept in pinned host memory ("DualDecoder: Accelerate Long Context LLM
Inference by Predictive Prefetch", §4.1, §5.2-§5.4).  Shapes follow a Llama-3-8B
decode layer (32 query / 8 KV heads, d = 128) and four stress variants; the
pages themselves publish no shapes (their accuracy experiments use RULER
needle-in-a-haystack with a sparse budget of 1024 entries, Table 1), so these
synthetic workloads stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int          # tokens per landmark block (B)
    top_k: int               # selected blocks per (request, KV head)
    window: int              # GPU-resident recent window (W tokens)
    n_layers: int
    ctx: Tuple[int, int]     # context length range [lo, hi] (lo == hi: fixed)
    key_dist: str = "normal"          # normal | channel_scaled | clustered
    plant: Optional[str] = None       # None | blocks | token_runs
    n_planted: int = 0
    plant_beta: float = 0.0
    spec_sigma: Optional[float] = None  # speculative query noise (None: no speculation)
    n_centroids: int = 0
    centroid_sigma: float = 0.0
    lowrank_rank: int = 0                # key_dist "lowrank": rank of the synthetic keys

    @property
    def group_size(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# Speculative-query noise of the long-context workload: q_spec = q + sigma * N(0,1),
# sigma chosen so the mean overlap |T n P| / k is about 0.88, the retrieval-index
# prediction accuracy DualDecoder reports (abstract; Fig. 16).  Calibrated by
# tests/golden/calibrate_spec_noise.py with the oracle's scoring.
SPEC_SIGMA_88 = 0.138

WORKLOADS = {
    # 1 request, 8 q / 2 KV heads, d 64, context 4096, block 16 (252 candidate
    # blocks after the 64-token window), top-16, 8 planted high-score blocks per KV head.
    "tiny": Workload("tiny", 1, 8, 2, 64, 16, 16, 64, 1, (4096, 4096),
                     key_dist="normal", plant="blocks", n_planted=8, plant_beta=2.0),
    # Llama-3-8B decode layer shape, 32 layers cycled through the ping-pong buffer.
    "llama3_8b_decode": Workload("llama3_8b_decode", 16, 32, 8, 128, 32, 64, 512, 32,
                                 (32768, 32768), key_dist="channel_scaled"),
    # Long context with prediction: ragged lengths, speculative query, urgent misses.
    "long_ctx_predict": Workload("long_ctx_predict", 64, 32, 8, 128, 32, 128, 512, 1,
                                 (65536, 131072), key_dist="normal", spec_sigma=SPEC_SIGMA_88),
    # Wide budget: 64 q / 8 KV heads, 256K context, block 64, 4096-token budget,
    # keys clustered around 32 Gaussian centroids (sigma 0.3) per (request, KV head).
    "wide_budget": Workload("wide_budget", 8, 64, 8, 128, 64, 64, 512, 1, (262144, 262144),
                            key_dist="clustered", n_centroids=32, centroid_sigma=0.3),
    # Fragmentation stress: token-granular blocks, top-2048 tokens per KV head,
    # planted as 60% isolated tokens and 40% in runs of 2..64.
    "fragmentation": Workload("fragmentation", 32, 32, 8, 128, 1, 2048, 512, 1, (65536, 65536),
                              key_dist="normal", plant="token_runs", n_planted=2048,
                              plant_beta=12.0),
    # Low-rank keys with prediction (DualDecoder §5.3: low-rank key reconstruction
    # for missed entries): the long-context shape at half the batch with rank-32
    # keys, so missed keys can be rebuilt on the GPU instead of fetched.
    "lowrank_predict": Workload("lowrank_predict", 32, 32, 8, 128, 32, 128, 512, 1, (65536, 131072),
                                key_dist="lowrank", lowrank_rank=32, spec_sigma=SPEC_SIGMA_88),
}

ORDER = ["tiny", "llama3_8b_decode", "long_ctx_predict", "wide_budget", "fragmentation", "lowrank_predict"]
