"""Placement of whole matrices on the GPUs of one node.

Every (matrix, block) unit of the optimizer is independent once its block
moments are known ("Dobb", Abstract: the update is computed locally within
each block; thelatestinai.com page, Table 3: the update needs no
communication), so a multi-GPU run places whole matrices on ranks and each
rank runs its own optimizer handle over its matrices, with no collective on
the data path.  The placement balances an estimate of each matrix's device
time per step: the update and moment streams (bytes per parameter and per
token row) plus the amortised refresh (k^3 per block every T steps).
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def matrix_cost(m: int, n: int, B: int, tokens: int, refresh_period: int) -> float:
    """Relative device time of one matrix per step (bytes-equivalent units)."""
    k = n // B
    update = 14.0 * m * n                     # G, M r/w, W r/w at bf16 parameters
    moments = 2.0 * tokens * n                # activation read
    refresh = 9.0 * B * k ** 3 / max(refresh_period, 1) / 10.0   # ~10 flop per byte balance
    return update + moments + refresh


def partition_matrices(shapes: Sequence[Tuple[int, int]], B: int, world: int, tokens: int = 8192,
                       refresh_period: int = 10) -> List[List[int]]:
    """Longest-processing-time placement of the matrices on `world` ranks.
    Returns, per rank, the sorted indices of the matrices it owns; every
    matrix is owned by exactly one rank, and the result depends only on the
    arguments (every rank computes the same placement)."""
    if world < 1:
        raise ValueError("world must be >= 1")
    cost = [(matrix_cost(m, n, B, tokens, refresh_period), i) for i, (m, n) in enumerate(shapes)]
    cost.sort(key=lambda c: (-c[0], c[1]))
    load = [0.0] * world
    owned: List[List[int]] = [[] for _ in range(world)]
    for c, i in cost:
        r = min(range(world), key=lambda j: (load[j], j))
        load[r] += c
        owned[r].append(i)
    return [sorted(o) for o in owned]
