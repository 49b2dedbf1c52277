"""z-slab decomposition across ranks: which planes each rank stores, and its ghost exchange.

The grid is cut along z into one slab per rank, the same partition as the library's
stencil_slabs_* calls: slab k owns the global planes [o_k, o_k+1), o_k = floor(k*nz/P),
and stores [max(0, o_k - R), min(nz, o_k+1 + R)), its owned planes plus up to R ghost
planes per side.  Before each sweep or step every rank sends its R owned planes next to
each cut to the neighbour across it and receives its ghost planes in return: two
point-to-point messages per cut and direction, no collective.  The sweep itself is the
library's stencil_apply on each rank's slab array (its ghost planes are slab-local shell).

Only the plane bookkeeping and the message pattern live here; torch.distributed moves
the bytes (gloo for CPU tensors).
"""
from __future__ import annotations


def partition(nz: int, nslabs: int, radius: int) -> list[dict]:
    """Per slab: stored planes [begin, end) and owned planes [own_begin, own_end)."""
    if nslabs < 1 or nz // nslabs < radius:
        raise ValueError(f"{nslabs} slabs of {nz} planes: every slab must own at least {radius} planes")
    own = [nz * k // nslabs for k in range(nslabs + 1)]
    return [{"begin": max(0, own[k] - radius), "end": min(nz, own[k + 1] + radius),
             "own_begin": own[k], "own_end": own[k + 1]} for k in range(nslabs)]


def ghost_messages(nz: int, nslabs: int, radius: int) -> list[dict]:
    """The exchange as messages: R planes from slab `src` (its local planes
    [src_plane, src_plane + R)) into slab `dst` (local planes [dst_plane, ...))."""
    parts = partition(nz, nslabs, radius)
    msgs = []
    for c in range(1, nslabs):
        lo, hi = parts[c - 1], parts[c]
        cut = hi["own_begin"]
        msgs.append({"src": c, "src_plane": cut - hi["begin"], "dst": c - 1, "dst_plane": cut - lo["begin"],
                     "planes": radius})
        msgs.append({"src": c - 1, "src_plane": cut - radius - lo["begin"], "dst": c,
                     "dst_plane": cut - radius - hi["begin"], "planes": radius})
    return msgs


def exchange_ghosts(dist, slab, rank: int, world: int, nz: int, radius: int, group=None) -> None:
    """Fill this rank's ghost planes from its neighbours.  `slab` is this rank's stored
    array, shape (end - begin, ny, nx), a contiguous torch tensor; rank k holds slab k."""
    reqs = []
    for m in ghost_messages(nz, world, radius):
        if m["src"] == rank:
            buf = slab[m["src_plane"]:m["src_plane"] + m["planes"]].contiguous()
            reqs.append(dist.isend(buf, dst=m["dst"], group=group))
        elif m["dst"] == rank:
            view = slab[m["dst_plane"]:m["dst_plane"] + m["planes"]]
            reqs.append((dist.irecv(view, src=m["src"], group=group), view))
    for r in reqs:
        (r[0] if isinstance(r, tuple) else r).wait()
