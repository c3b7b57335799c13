"""Grouped program -> tile ordering, written from its description -- TEST INFRASTRUCTURE ONLY.

Page "I3. Fuse a GEMM epilogue and change tile scheduling", section "Tiles and
grouped ownership": a one-dimensional program id walks bands of GROUP M-tiles;
inside a band the M index moves fastest; the last band may hold fewer than
GROUP M-tiles, so the within-band remainder and quotient are taken with
actual_group = min(GROUP, tiles_m - first_m).  GROUP = 1 is row-major order.
"""
from __future__ import annotations


def tile_of(pid: int, tiles_m: int, tiles_n: int, group: int) -> tuple[int, int]:
    """Return (m_tile, n_tile) owned by program ``pid``."""
    band = group * tiles_n                  # programs per band of GROUP M-tiles
    first_m = (pid // band) * group         # first M-tile of this band
    actual_group = min(group, tiles_m - first_m)
    within = pid % band
    m_tile = first_m + within % actual_group
    n_tile = within // actual_group
    return m_tile, n_tile


def order(tiles_m: int, tiles_n: int, group: int) -> list[tuple[int, int]]:
    """The whole sequence of tiles for pids 0 .. tiles_m*tiles_n - 1."""
    return [tile_of(p, tiles_m, tiles_n, group) for p in range(tiles_m * tiles_n)]
