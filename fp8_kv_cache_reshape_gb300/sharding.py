"""Head-sharded decode across ranks: which KV heads (and so which query heads
and which pages' bytes) each rank owns.

"kv-cache-quantization-fp8-scale-granularity" (the inference-research note)
describes the KV cache as partitioned across tensor-parallel ranks.  Decode
attention has no exchange step under that partition: query head h reads only
KV head h / g (g = Hq / Hkv, contiguous groups), so a rank that holds a
contiguous range of KV heads -- their K and V pages and per-head scales --
and the query heads of those groups computes exactly the output rows of
those query heads, with the same kernels and no collective.  The full
[B][Hq][D] output is the concatenation of the ranks' [B][Hq / N][D] slices
along the head axis (in a model, the following output projection is where a
tensor-parallel reduction would sit).

This module is host logic only (no device code, no torch): it checks that
the partition exists and gives each rank its head ranges.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class HeadShard:
    """One rank's part: KV heads [kv0, kv1) and query heads [q0, q1)."""
    rank: int
    world: int
    kv0: int
    kv1: int
    q0: int
    q1: int

    @property
    def kv_heads(self) -> int:
        return self.kv1 - self.kv0

    @property
    def q_heads(self) -> int:
        return self.q1 - self.q0


def kv_head_shard(q_heads: int, kv_heads: int, world: int, rank: int) -> HeadShard:
    """Rank `rank` of `world` owns KV heads [rank * Hkv / N, (rank + 1) * Hkv / N)
    and their query-head groups.  Raises ValueError unless Hq % Hkv == 0 and
    Hkv % N == 0 (every rank gets the same number of whole groups)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    if q_heads < 1 or kv_heads < 1 or q_heads % kv_heads:
        raise ValueError(f"query heads {q_heads} are not whole groups of {kv_heads} KV heads")
    if kv_heads % world:
        raise ValueError(f"{kv_heads} KV heads do not split evenly over {world} ranks")
    g = q_heads // kv_heads
    per = kv_heads // world
    kv0 = rank * per
    return HeadShard(rank, world, kv0, kv0 + per, kv0 * g, (kv0 + per) * g)


def all_shards(q_heads: int, kv_heads: int, world: int) -> list:
    return [kv_head_shard(q_heads, kv_heads, world, r) for r in range(world)]
