"""Column-tile sharding of one tiled weight over ranks (host logic only, no device code).

The tiled layout ("Hexagon backend developer details", "Tiled Weight Formats", "Tile Dimensions and
Grid Layout") stores tile (ct, kt) at (ct * n_k_tiles + kt) * tile_size, so a contiguous range of
column tiles is a contiguous byte range of the weight and produces a contiguous range of output
columns with no reduction across ranks.  A rank runs the ordinary matmul on its slice: the tiles
at `byte_offset`, N = `n_local`, and y offset by `n0` columns with the full ldy.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Shard:
    rank: int
    world: int
    ct0: int            # first column tile of this rank
    ct1: int            # one past the last
    n0: int             # first output column
    n_local: int        # output columns of this rank (0 when the rank has no tile)
    byte_offset: int    # offset of tile (ct0, 0) in the tiled weight
    byte_len: int       # bytes of this rank's tiles


TILE_BYTES = {"q4_0": 576, "iq4_nl": 576, "q8_0": 1088, "mxfp4": 544, "q4_1": 640, "q4_k": 640}


def tile_bytes(type_: str) -> int:
    return TILE_BYTES[type_]


def col_tile_range(n_col_tiles: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced split: the first n_col_tiles % world ranks take one tile more."""
    if world <= 0 or not 0 <= rank < world or n_col_tiles < 0:
        raise ValueError("bad rank/world")
    base, extra = divmod(n_col_tiles, world)
    ct0 = rank * base + min(rank, extra)
    return ct0, ct0 + base + (1 if rank < extra else 0)


def shard(type_: str, K: int, N: int, rank: int, world: int) -> Shard:
    if K <= 0 or K % 32 or N <= 0:
        raise ValueError("K must be a positive multiple of 32 and N positive")
    nkt, nct = K // 32, (N + 31) // 32
    ct0, ct1 = col_tile_range(nct, rank, world)
    n0 = ct0 * 32
    n_local = max(0, min(N, ct1 * 32) - n0)
    tb = tile_bytes(type_)
    return Shard(rank, world, ct0, ct1, n0, n_local, ct0 * nkt * tb, (ct1 - ct0) * nkt * tb)
