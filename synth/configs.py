"""The five SFI decode-attention workloads, as plain data.

Each workload is one attention layer stack decoded for a number of steps after a
prefill: GQA layers with 4 query heads per kv head and head dim 128 (Llama-3-8B's 32 query
and 8 kv heads in all but the 4K case), a sparse budget of sinks + recent window +
selected positions, and a seeded boundary mask that decides the slow steps.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx: int                 # prefill length (upper end for ragged batches)
    ctx_lo: int              # lower end for ragged batches (== ctx otherwise)
    steps: int
    n_sink: int
    n_window: int
    n_select: int
    key_model: str           # 'hh' (planted heavy hitters) or 'zipf' (Zipf key-norm boost)
    mask_kind: str           # 'periodic' or 'geometric'
    mask_param: float
    per_seq_mask: bool = False
    page_size: int = 0       # 0 = contiguous cache, 16 = paged
    drift: bool = False      # heavy hitters re-seeded at each boundary
    trigger: str = "mask"    # 'mask': seeded boundary mask; 'tokens': trigger tokens in a
                             # seeded token stream (mean span mask_param) decide the slow steps
    lam: float = 0.1         # fusion weight of the prior
    t_max: int = 64          # forced refresh after this many steps without a slow step
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def prior_tau(self) -> int:
        return self.n_window

    @property
    def capacity(self) -> int:
        """Positions per (layer, sequence, kv head) the cache must hold."""
        return self.ctx + self.steps

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "gqa4_ctx4k_hh": Workload(
        name="gqa4_ctx4k_hh", n_layers=1, batch=1, n_q_heads=8, n_kv_heads=2, head_dim=128,
        ctx=4096, ctx_lo=4096, steps=32, n_sink=4, n_window=64, n_select=256,
        key_model="hh", mask_kind="periodic", mask_param=16, seed=0x5F1000 + 1),
    "llama8b_ctx32k_b4": Workload(
        name="llama8b_ctx32k_b4", n_layers=1, batch=4, n_q_heads=32, n_kv_heads=8, head_dim=128,
        ctx=32768, ctx_lo=32768, steps=256, n_sink=4, n_window=64, n_select=1980,
        key_model="zipf", mask_kind="geometric", mask_param=18, seed=0x5F1000 + 2),
    "llama8b_ctx128k_l32": Workload(
        name="llama8b_ctx128k_l32", n_layers=32, batch=1, n_q_heads=32, n_kv_heads=8,
        head_dim=128, ctx=131072, ctx_lo=131072, steps=128, n_sink=4, n_window=64,
        n_select=1980, key_model="zipf", mask_kind="geometric", mask_param=18,
        seed=0x5F1000 + 3),
    "ragged_paged_b32": Workload(
        name="ragged_paged_b32", n_layers=1, batch=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
        ctx=32768, ctx_lo=8192, steps=128, n_sink=4, n_window=64, n_select=956,
        key_model="zipf", mask_kind="geometric", mask_param=15, per_seq_mask=True,
        page_size=16, seed=0x5F1000 + 4),
    "longcot_ctx128k_b8_l32": Workload(
        name="longcot_ctx128k_b8_l32", n_layers=32, batch=8, n_q_heads=32, n_kv_heads=8,
        head_dim=128, ctx=131072, ctx_lo=131072, steps=512, n_sink=4, n_window=128,
        n_select=1916, key_model="hh", mask_kind="geometric", mask_param=24, drift=True,
        seed=0x5F1000 + 5),
    # the 32K batch-4 shape with the trigger rule itself: every sequence generates its own
    # token stream, and a slow step follows a trigger token ('.', '?', '!', newline)
    "llama8b_ctx32k_b4_tok": Workload(
        name="llama8b_ctx32k_b4_tok", n_layers=1, batch=4, n_q_heads=32, n_kv_heads=8,
        head_dim=128, ctx=32768, ctx_lo=32768, steps=256, n_sink=4, n_window=64, n_select=1980,
        key_model="zipf", mask_kind="geometric", mask_param=18, per_seq_mask=True,
        trigger="tokens", seed=0x5F1000 + 6),
}

ORDER = ["gqa4_ctx4k_hh", "llama8b_ctx32k_b4", "llama8b_ctx128k_l32", "ragged_paged_b32",
         "longcot_ctx128k_b8_l32"]
