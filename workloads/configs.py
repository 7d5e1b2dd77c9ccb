"""The named decode and chunk workloads and the spec type for custom ones.

Shapes follow the decode configurations the paged-attention pages motivate:
GQA head groups ("vLLM 0.7.2深度解析" §2.2), block sizes 16 and 32 (§2.1 of the
same page; "vLLM 0.5 深度解析" §3.1), a 4K sliding window (§2.3 of the 0.7.2
page), shared prefixes (§2.1) and an FP8 e4m3 cache (§2.2).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Spec:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str = "bf16"            # q and the 16-bit K/V values: "f16" | "bf16"
    kv_fp8: bool = False           # store the cache as e4m3 with per-tensor scales
    window: int = 0                # sliding window (0: off)
    # sequence lengths: explicit tuple, or a distribution
    seq_lens: tuple | None = None
    len_dist: tuple = ("uniform", 1, 200)   # ("uniform"|"loguniform", lo, hi)
    long_seqs: tuple = ()          # extra fixed lengths placed first (skewed batches)
    shared_prefix: int = 0         # tokens shared by every sequence (multiple of block_size)
    max_len: int | None = None     # sizes max_blocks_per_seq; default: the distribution's max
    pool_blocks: int | None = None # explicit pool size; default ceil(pool_factor * need)
    pool_factor: float = 1.2
    new_tokens: bool = True        # the last position(s) of each sequence are written by reshape
    num_queries: int = 1           # query tokens per sequence (a chunk at its last positions)
    seed: int = 0
    scale: float | None = None     # default head_dim ** -0.5
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else self.head_dim ** -0.5

    def with_(self, **kw) -> "Spec":
        return replace(self, **kw)


def _seed(index: int) -> int:
    return 267 * 1000 + index


CONFIGS: dict[str, Spec] = {
    "tiny": Spec("tiny", batch=4, num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                 dtype="f16", len_dist=("uniform", 1, 200), pool_blocks=64, seed=_seed(1)),
    "llama8b": Spec("llama8b", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
                    block_size=16, dtype="bf16", len_dist=("uniform", 512, 4096),
                    pool_factor=1.2, seed=_seed(2)),
    "long_skew": Spec("long_skew", batch=8, num_q_heads=64, num_kv_heads=8, head_dim=128,
                      block_size=32, dtype="bf16", long_seqs=(131072,),
                      len_dist=("uniform", 256, 2048), max_len=131072, pool_factor=1.2,
                      seed=_seed(3)),
    "prefix_window": Spec("prefix_window", batch=128, num_q_heads=32, num_kv_heads=8,
                          head_dim=128, block_size=16, dtype="bf16", window=4096,
                          shared_prefix=2048, len_dist=("uniform", 128, 30000),
                          pool_factor=1.2, seed=_seed(4)),
    "fp8": Spec("fp8", batch=256, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                dtype="bf16", kv_fp8=True, len_dist=("loguniform", 1024, 8192),
                pool_factor=1.2, seed=_seed(5)),
    # chunked queries (pa_prefill_chunk): T query tokens per sequence at its
    # last T positions, causal within the chunk
    "verify4_llama8b": Spec("verify4_llama8b", batch=64, num_q_heads=32, num_kv_heads=8,
                            head_dim=128, block_size=16, dtype="bf16",
                            len_dist=("uniform", 512, 4096), num_queries=4, pool_factor=1.2,
                            seed=_seed(6)),
    "prefill_chunk512": Spec("prefill_chunk512", batch=8, num_q_heads=32, num_kv_heads=8,
                             head_dim=128, block_size=16, dtype="bf16",
                             len_dist=("uniform", 512, 8192), num_queries=512, pool_factor=1.2,
                             seed=_seed(7)),
    "prefill_chunk512_fp8": Spec("prefill_chunk512_fp8", batch=8, num_q_heads=32, num_kv_heads=8,
                                 head_dim=128, block_size=16, dtype="bf16", kv_fp8=True,
                                 len_dist=("uniform", 512, 8192), num_queries=512,
                                 pool_factor=1.2, seed=_seed(8)),
}


def get_config(name: str) -> Spec:
    return CONFIGS[name]
