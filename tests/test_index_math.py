"""Host checks of the kernels' index arithmetic (no GPU): the same formulas
as the CUDA sources, evaluated over the shapes the kernels see, so that a
change to one of them that breaks coverage or bounds fails here first."""

import pytest


def xpad(c):
    """Decode GEMV: staged activation chunk c sits at c + c / 8."""
    return c + (c >> 3)


@pytest.mark.parametrize("kseg,cpl", [(128, 4), (64, 2)])      # 4-bit formats, FP8
def test_gemv_activation_chunks_from_one_base_per_segment(kseg, cpl):
    """The lane reads chunk j of segment s at base(s, t) + j, with
    base = (s_lo + s) * (KSEG/8 + KSEG/64) + xpad(t * CPL): that must be
    xpad of the chunk's own index for every lane, segment and j, and the
    padded positions must be distinct (no two chunks share a slot)."""
    pad_seg = kseg // 8 + kseg // 64
    seen = set()
    for seg in range(40):
        for t in range(4):
            for j in range(cpl):
                c = seg * (kseg // 8) + t * cpl + j
                assert seg * pad_seg + xpad(t * cpl) + j == xpad(c)
                seen.add(xpad(c))
    nchunk = 40 * (kseg // 8)
    assert len(seen) == nchunk
    assert max(seen) < nchunk + nchunk // 8          # fits the host's row pitch


@pytest.mark.parametrize("want", [1, 2])
def test_gemv_activation_reads_are_bank_conflict_free(want):
    """The 16-byte reads of one quarter-warp (lanes 8h .. 8h+7: activation rows
    2h, 2h+1 and lane positions t = 0..3) fall in 8 distinct 4-bank groups
    with the host's row pitch (ncp = want mod 8; 2 for 4-bit, 1 for FP8)."""
    kseg, cpl = (128, 4) if want == 2 else (64, 2)
    ncp = 8 * 37 + want
    for seg in range(6):
        for h in range(4):
            groups = set()
            for lane in range(8 * h, 8 * h + 8):
                g, t = lane >> 2, lane & 3
                c = seg * (kseg // 8) + t * cpl
                groups.add((g * ncp + xpad(c)) % 8)
            assert len(groups) == 8


def tile_origin(tile, tiles_t, tiles_w, group_t):
    """Prefill raster: group_t token tiles share a group; tile -> (token tile, channel tile)."""
    per_group = group_t * tiles_w
    grp = tile // per_group
    first_t = grp * group_t
    gsize = min(group_t, tiles_t - first_t)
    within = tile - grp * per_group
    return first_t + within % gsize, within // gsize


@pytest.mark.parametrize("group_t", [1, 2, 8])
@pytest.mark.parametrize("tiles_t,tiles_w", [(32, 112), (32, 32), (3, 5), (1, 7), (17, 9)])
def test_prefill_raster_covers_every_tile_once(group_t, tiles_t, tiles_w):
    seen = {tile_origin(i, tiles_t, tiles_w, group_t) for i in range(tiles_t * tiles_w)}
    assert seen == {(a, b) for a in range(tiles_t) for b in range(tiles_w)}
