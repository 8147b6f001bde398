"""Work partition of the attention forward over several GPUs (one process per GPU).

A unit is one (batch index, key/value head): the pooling, mask rows and attention rows of the
query heads that share that key/value head read nothing of any other unit, so the units can be
spread over ranks with no exchange between them.  A rank runs the library's calls on views of
its units (the calls accept strided tensors), and the outputs of all ranks together are the
single-GPU outputs; only a caller who wants every head on one GPU gathers them afterwards."""
from __future__ import annotations

from typing import List, Tuple


def units(B: int, Hkv: int) -> List[Tuple[int, int]]:
    """Every (b, kvh) unit, batch-major."""
    return [(b, g) for b in range(B) for g in range(Hkv)]


def shard_units(B: int, Hkv: int, world: int, rank: int) -> List[Tuple[int, int]]:
    """The units of one rank: a contiguous run of the batch-major list, the runs differing in
    length by at most one unit."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("rank %d of a world of %d" % (rank, world))
    u = units(B, Hkv)
    base, extra = divmod(len(u), world)
    start = rank * base + min(rank, extra)
    return u[start:start + base + (1 if rank < extra else 0)]


def unit_heads(unit: Tuple[int, int], Hq: int, Hkv: int) -> Tuple[int, slice, int]:
    """(b, query-head slice, kv head) of a unit: query heads kvh * G .. (kvh + 1) * G - 1, G = Hq / Hkv."""
    b, kvh = unit
    G = Hq // Hkv
    return b, slice(kvh * G, (kvh + 1) * G), kvh
