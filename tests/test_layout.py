"""Host-side checks of the code layout and of the shared-memory table layout
used by the list scan (restated from csrc/layout.cuh and csrc/scan.cuh)."""

import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def group_size(g, m):
    return min(32, m - 32 * g)


def stored_source_byte(lane, s, m):
    g0 = s & ~31
    return g0 + (lane + (s - g0)) % group_size(s >> 5, m)


def stored_byte_offset(lane, s, m):
    nfull = m >> 4
    c = s >> 4
    if c < nfull:
        return c * 512 + lane * 16 + (s & 15)
    r = m & 15
    return nfull * 512 + lane * r + (s - (nfull << 4))


@pytest.mark.parametrize("m", list(range(4, 65, 4)))
def test_block_layout_is_a_bijection(m):
    offs = set()
    for lane in range(32):
        src = [stored_source_byte(lane, s, m) for s in range(m)]
        assert sorted(src) == list(range(m))  # every code byte stored once
        for s in range(m):
            o = stored_byte_offset(lane, s, m)
            assert 0 <= o < 32 * m
            offs.add(o)
    assert len(offs) == 32 * m  # no two stored bytes share a position


def lut_table_of_column(col, g, m):
    return 32 * g + col % group_size(g, m)


@pytest.mark.parametrize("m", [4, 8, 12, 16, 24, 32, 40, 64])
def test_scan_reads_the_right_table_without_bank_conflicts(m):
    """At step s of group g lane i reads column i + s of row e. That column
    must hold the table of the code byte stored at position 32g + s, and the
    32 lanes must hit 32 distinct banks for any code bytes."""
    rng = np.random.default_rng(m)
    for s_all in range(m):
        g, s = s_all >> 5, s_all & 31
        banks = set()
        for lane in range(32):
            col = lane + s
            assert col < 64
            assert lut_table_of_column(col, g, m) == stored_source_byte(lane, s_all, m)
            e = int(rng.integers(0, 256))
            word = g * 256 * 64 + e * 64 + col
            banks.add(word % 32)
        assert len(banks) == 32


def _worst_conflicts(entry_bytes):
    """Worst case over all lane->entry assignments of one look-up instruction
    on a plain 256-entry table (entry e at byte e*entry_bytes): the number of
    distinct 4-byte words in the busiest bank, minus one."""
    words_per_bank = {}
    for e in range(256):
        w = e * entry_bytes // 4
        words_per_bank.setdefault(w % 32, set()).add(w)
    return max(len(v) for v in words_per_bank.values()) - 1


def test_plain_table_conflicts_match_the_pages():
    rows = []
    with open(os.path.join(GOLDEN, "lut_bank_conflicts.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    for entry_bytes, worst in rows:
        assert _worst_conflicts(entry_bytes) == worst


@pytest.mark.parametrize("gs", [4, 8, 16, 32])
def test_table_build_stores_are_conflict_free(gs):
    """Build: lane -> (jj = lane % gs, qq = lane // gs), store s writes copy
    (s + qq) % (64/gs) of its table's columns."""
    reps = 64 // gs
    for it in range(0, 256 * gs, 32):
        for s in range(reps):
            banks = set()
            for lane in range(32):
                jj, qq = lane % gs, lane // gs
                e = (it + lane) // gs
                col = jj + gs * ((s + qq) % reps)
                assert col % gs == jj
                banks.add((e * 64 + col) % 32)
            assert len(banks) == 32
