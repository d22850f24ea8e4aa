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


@pytest.mark.parametrize("nseg", [1, 4, 7, 8, 32, 112, 224])
@pytest.mark.parametrize("ks", [1, 2, 4, 8])
@pytest.mark.parametrize("kw", [1, 2, 4, 8])
def test_gemv_k_split_partitions_the_segments(nseg, ks, kw):
    """K segments split over the ks CTAs of a cluster, then over the kw warps
    of a row group (the GEMV's seg_lo/seg_hi and s_lo/s_hi): every segment
    exactly once, in order."""
    got = []
    for kr in range(ks):
        seg_lo, seg_hi = nseg * kr // ks, nseg * (kr + 1) // ks
        n_cta = seg_hi - seg_lo
        for w in range(kw):
            s_lo, s_hi = n_cta * w // kw, n_cta * (w + 1) // kw
            got.extend(seg_lo + s for s in range(s_lo, s_hi))
    assert got == list(range(nseg))


@pytest.mark.parametrize("rows_cta", [16, 32, 64, 128])
@pytest.mark.parametrize("ks", [1, 2, 4, 8])
def test_gemv_cluster_epilogue_rows(rows_cta, ks):
    """Each CTA of a cluster finishes rows_cta / ks rows of the shared tile:
    together every row once."""
    rows_per = rows_cta // ks
    got = sorted(kr * rows_per + r for kr in range(ks) for r in range(rows_per))
    assert got == list(range(rows_cta))


@pytest.mark.parametrize("ntiles_total", [1, 112, 151, 152, 153, 448, 1024])
def test_persistent_tile_lists_cover_every_tile(ntiles_total):
    """Persistent kernels: CTA b of a grid of min(tiles, 152) takes tiles
    b, b + grid, ...; the count each CTA computes for itself adds up."""
    grid = min(ntiles_total, 152)
    got = []
    for b in range(grid):
        ntiles = (ntiles_total - b + grid - 1) // grid
        got.extend(b + i * grid for i in range(ntiles))
    assert sorted(got) == list(range(ntiles_total))
