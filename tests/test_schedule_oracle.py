"""Pins for the grouped tile ordering of the oracle (CPU only)."""
import random

from conftest import read_golden
from oracle import schedule


def test_six_program_table():
    # "I3. Fuse a GEMM epilogue and change tile scheduling", "Tiles and grouped ownership".
    g = read_golden("grouped_order_3x2_g2.txt")
    tm, tn, grp = int(g["tiles_m"]), int(g["tiles_n"]), int(g["group"])
    want = [tuple(int(x) for x in g[str(p)].split(",")) for p in range(tm * tn)]
    assert schedule.order(tm, tn, grp) == want


def test_group_one_is_row_major():
    assert schedule.order(4, 3, 1) == [(m, n) for m in range(4) for n in range(3)]


def test_group_at_least_tiles_m_is_column_major():
    assert schedule.order(3, 4, 8) == [(m, n) for n in range(4) for m in range(3)]


def test_incomplete_final_group_is_a_bijection():
    # the page warns that using GROUP unconditionally duplicates or loses tiles
    for tm, tn, grp in [(3, 2, 2), (5, 7, 4), (9, 1, 8), (1, 9, 8), (64, 56, 8), (8, 85, 3)]:
        seen = schedule.order(tm, tn, grp)
        assert sorted(seen) == [(m, n) for m in range(tm) for n in range(tn)]


def test_random_shapes_bijection():
    rnd = random.Random(5)
    for _ in range(200):
        tm, tn, grp = rnd.randint(1, 30), rnd.randint(1, 30), rnd.randint(1, 12)
        assert len(set(schedule.order(tm, tn, grp))) == tm * tn


def test_unconditional_group_loses_tiles():
    # negative control: the mistake the page warns about is caught by the bijection check
    def bad(pid, tm, tn, grp):
        band = grp * tn
        first = (pid // band) * grp
        return first + (pid % band) % grp, (pid % band) // grp
    tiles = [bad(p, 3, 2, 2) for p in range(6)]
    assert sorted(tiles) != [(m, n) for m in range(3) for n in range(2)]
