"""CPU enumeration of the pre-scaled kernel's B-fragment layout in shared
memory (col_slot / frag_off in quantized_gemv_tq2_gb300/csrc/tq2_matvec_ps.cu).

The expressions are read from the kernel source and evaluated here, so a
change to the layout is checked by these properties, for M = 1..16:
  * per 256-block the entries (n-tile, word jw, half h, quad t, column g)
    fill the block's 512*M bytes exactly once (a bijection of 16-byte slots);
  * a full n-tile (8 columns) is conflict-free for the MMA reads (8 lanes of
    a load phase: g in {2q, 2q+1}, t in 0..3, one jw and h) and for the
    staging writes (8 lanes of a store phase: t in {2p, 2p+1}, jw in 0..3,
    one column g and half h): 8 distinct 16-byte bank groups each;
  * a partial n-tile (Mt < 8 columns) keeps the plain layout: its load
    phases are at most 2-way (1-way for Mt = 1, 2, 6; 2-way for 3, 4, 5, 7)
    and its store phases 4-way.
Shared memory serves a 16-byte access for 8 lanes per wavefront; lanes of a
phase that hit the same 16-byte slot of a 128-byte row are one access (a
broadcast), distinct slots in the same bank group conflict.
"""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "quantized_gemv_tq2_gb300", "csrc", "tq2_matvec_ps.cu")


def _layout():
    src = open(SRC).read()
    m_sw = re.search(r"const int sw = ([^;]+);", src)
    m_ret = re.search(r"return t \* Mt \+ \(Mt == 8 \? \(g \^ sw\) : g\);", src)
    m_off = re.search(r"const int Mt = min\(8, M - 8 \* nt\);\s*return \(uint32_t\)\(([^;]+)\);", src)
    assert m_sw and m_ret and m_off, "the layout functions changed: update this enumeration"
    sw_expr = m_sw.group(1)
    off_expr = m_off.group(1)

    def col_slot(t, g, jw, Mt):
        sw = eval(sw_expr, {}, {"t": t, "jw": jw})
        return t * Mt + ((g ^ sw) if Mt == 8 else g)

    def frag_off(bx, nt, jw, h, t, g, M):
        Mt = min(8, M - 8 * nt)
        return eval(off_expr, {"col_slot": col_slot},
                    {"bx": bx, "nt": nt, "jw": jw, "h": h, "t": t, "g": g, "M": M, "Mt": Mt})

    return col_slot, frag_off


def _degree(addrs):
    """Wavefronts needed for one 8-lane phase of 16-byte accesses: distinct
    addresses per 16-byte bank group (addr / 16 mod 8), maximised."""
    groups = {}
    for a in set(addrs):
        groups.setdefault((a // 16) % 8, set()).add(a)
    return max(len(v) for v in groups.values())


@pytest.mark.parametrize("M", range(1, 17))
def test_block_layout_is_a_bijection(M):
    _, frag_off = _layout()
    NT = (M + 7) // 8
    seen = []
    for nt in range(NT):
        Mt = min(8, M - 8 * nt)
        for jw in range(4):
            for h in range(2):
                for t in range(4):
                    for g in range(Mt):
                        seen.append(frag_off(0, nt, jw, h, t, g, M))
    assert all(o % 16 == 0 for o in seen)
    assert sorted(seen) == list(range(0, 512 * M, 16)), M
    # the next block starts where this one ends
    assert frag_off(1, 0, 0, 0, 0, 0, M) == 512 * M


@pytest.mark.parametrize("M", range(1, 17))
def test_access_phases(M):
    _, frag_off = _layout()
    NT = (M + 7) // 8
    for nt in range(NT):
        Mt = min(8, M - 8 * nt)
        load_deg, store_deg = 1, 1
        # MMA reads: lane (g, t) = (lane >> 2, lane & 3); columns past M read column 0
        for jw in range(4):
            for h in range(2):
                for q in range(4):
                    addrs = []
                    for g in (2 * q, 2 * q + 1):
                        gsel = g if 8 * nt + g < M else 0
                        for t in range(4):
                            addrs.append(frag_off(0, nt, jw, h, t, gsel, M))
                    load_deg = max(load_deg, _degree(addrs))
        # staging writes: a half-warp's lane wi = 4 t + jw writes one column g
        for g in range(Mt):
            for h in range(2):
                for p in range(2):
                    addrs = [frag_off(0, nt, jw, h, t, g, M) for t in (2 * p, 2 * p + 1) for jw in range(4)]
                    store_deg = max(store_deg, _degree(addrs))
        if Mt == 8:
            assert load_deg == 1 and store_deg == 1, (M, nt, load_deg, store_deg)
        else:
            want_load = 1 if Mt in (1, 2, 6) else 2
            assert (load_deg, store_deg) == (want_load, 4), (M, nt, load_deg, store_deg)


def test_unswizzled_full_tile_would_conflict():
    """The property the swizzle exists for: with col = g a full n-tile gives
    4-way load and 8-way store phases (what ncu measured before it)."""
    col_slot, _ = _layout()
    Mt = 8

    def plain(jw, h, t, g):
        return jw * 128 * Mt + (h * 4 * Mt + t * Mt + g) * 16

    loads = max(_degree([plain(jw, h, t, g) for g in (2 * q, 2 * q + 1) for t in range(4)])
                for jw in range(4) for h in range(2) for q in range(4))
    stores = max(_degree([plain(jw, h, t, g) for t in (2 * p, 2 * p + 1) for jw in range(4)])
                 for g in range(8) for h in range(2) for p in range(2))
    assert (loads, stores) == (4, 8)
    # and the swizzled slot of a full tile is a permutation of the plain one per (t, jw)
    for t in range(4):
        for jw in range(4):
            assert sorted(col_slot(t, g, jw, 8) for g in range(8)) == [t * 8 + g for g in range(8)]
