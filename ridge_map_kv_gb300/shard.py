"""One fill sharded across GPUs by upper layer, with no data-path collective.

[RF] "Ridge map": every upper layer ℓ >= S has its own map A_ℓ, bias b_ℓ, norm and
projections, and a filled (row, layer) entry depends on x_S[row] and that layer's
weights alone. So the P = L - S upper layers split into contiguous blocks, one per
rank, the way pipeline-parallel serving places layers on GPUs: rank r holds the
maps, biases, gains and projections of its block and the cache slice of those
layers, reads the same x_S and exact-row mask as every other rank, and fills its
slice with one rf_fill_kv call. The ranks exchange nothing; together they write
every (row, layer) entry of the fill exactly once.

A rank's call describes its block as a fill of its own: L = its layer count and
S = 0, over a cache that holds just its layers (layer i of the local cache is
upper layer S + p0 + i of the model). Row partition, RoPE positions and every value
are those of the whole fill, because nothing in a row's computation depends on the
layer index beyond the choice of weights.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class LayerShard:
    rank: int
    world: int
    p0: int          # first upper layer of the block (0-based among the P upper layers)
    p1: int          # one past the last
    S: int           # the model's split layer: the block is model layers S + p0 .. S + p1 - 1

    @property
    def layers(self) -> int:
        return self.p1 - self.p0

    @property
    def model_layers(self) -> range:
        return range(self.S + self.p0, self.S + self.p1)


def layer_shard(P: int, S: int, world: int, rank: int) -> LayerShard:
    """Contiguous block of the P upper layers for ``rank`` of ``world``: the first
    P % world ranks take one layer more than the rest. A rank beyond P gets an
    empty block."""
    if world < 1 or not 0 <= rank < world or P < 0:
        raise ValueError(f"need world >= 1, 0 <= rank < world and P >= 0 (P={P}, world={world}, rank={rank})")
    base, extra = divmod(P, world)
    p0 = rank * base + min(rank, extra)
    p1 = p0 + base + (1 if rank < extra else 0)
    return LayerShard(rank, world, p0, p1, S)


def shard_desc_fields(fields: dict, shard: LayerShard) -> dict:
    """rf_fill_desc fields of a rank's block from those of the whole fill: L becomes
    the block's layer count and S becomes 0; everything else is unchanged."""
    out = dict(fields)
    out["L"] = shard.layers
    out["S"] = 0
    return out


def shard_weights(tensors: dict, shard: LayerShard) -> dict:
    """The rank's slices of the per-layer tensors (leading dimension P): maps A, b,
    gain, Wk, Wv, and the per-layer corrections v_scale and k_norm_gain when
    present. Other entries (x_S, mask) are shared and returned as they are."""
    per_layer = ("A", "b", "gain", "Wk", "Wv", "v_scale", "k_norm_gain")
    return {k: (v[shard.p0:shard.p1] if k in per_layer and v is not None else v) for k, v in tensors.items()}
