"""Shared-memory bank model (CPU). The rocm-libraries pull 10102 page counts
the LDS banks one wave's K read touches (Motivation); its printed table is
the golden fixture that pins the model here. The same model, redone for this
GPU (32 banks x 4 bytes; a 16-byte access per lane is served 8 lanes per
wavefront, one 128-byte row of banks), then checks that the layouts the
kernels use put the 8 rows of every wavefront in 8 distinct 16-byte bank
groups. The layout formulas below restate the kernels' address arithmetic
(GQA page tiles and padded rows, the GQA warp-merge rows, the MLA padded
rows, the prefill P tile)."""
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "lds_bank_table.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line:
            name, d, gr, gp, banks, lanes = line
            rows.append((name, int(d), int(gr), int(gp), int(banks), int(lanes)))
    return rows


def _amd_k_read(d, group_rows, group_pad):
    """Banks touched and the largest number of lane-dword accesses per bank
    for the page's QK read on gfx950 (64 banks x 4 bytes)."""
    per_bank = {}
    for lane in range(64):
        krow, col = lane % 32, (lane // 32) * 8
        group, sub = divmod(krow, group_rows)
        elem = group * (group_rows * d + group_pad) + sub * d + col
        dword = elem * 2 // 4
        for i in range(4):   # 8 bf16 = 4 dwords
            b = (dword + i) % 64
            per_bank[b] = per_bank.get(b, 0) + 1
    return len(per_bank), max(per_bank.values())


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_bank_model_reproduces_the_page_table(row):
    _, d, gr, gp, banks, lanes = row
    assert _amd_k_read(d, gr, gp) == (banks, lanes)


def _conflict_free(addrs16):
    """8-lane wavefronts of 16-byte accesses: 8 distinct 16-byte bank groups
    (32 banks x 4 bytes = 8 groups of 16 bytes)."""
    for w in range(0, len(addrs16), 8):
        groups = {(a // 16) % 8 for a in addrs16[w:w + 8]}
        if len(groups) != 8:
            return False
    return True


def _swizzled(r, c, slab_bytes):
    # 128-byte swizzle: 16-byte chunk c of row r, 64-element column slabs
    return (c >> 3) * slab_bytes + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4)


@pytest.mark.parametrize("d", [128, 256])
def test_gqa_tile_reads(d):
    # K (A of S^T): ldmatrix x4, lanes 0-15 rows 0-15 of chunk c, lanes 16-31
    # rows 0-15 of chunk c + 1; V^T: the transposing load, same row groups
    for c in range(d * 2 // 16 - 1):
        tile = [_swizzled(lane & 15, c + (lane >> 4), 2048) for lane in range(32)]
        assert _conflict_free(tile)
        pitch = d * 2 + 16   # padded rows (page sizes that are not page tiles)
        rows = [(lane & 15) * pitch + (c + (lane >> 4)) * 16 for lane in range(32)]
        assert _conflict_free(rows)
        unpadded = [(lane & 15) * d * 2 + (c + (lane >> 4)) * 16 for lane in range(32)]
        assert not _conflict_free(unpadded)   # why the pad is there


@pytest.mark.parametrize("d", [128, 256])
def test_gqa_merge_rows(d):
    # the mma C fragment stores: lane (g, t) writes row 2t (and 2t + 1) at
    # column g of the warp's merge rows; 4-byte stores, 32 lanes per wavefront
    for pad, ok in ((4, True), (0, False)):
        banks = {((2 * (lane & 3)) * (d + pad) + (lane >> 2)) % 32 for lane in range(32)}
        assert (len(banks) == 32) == ok


def test_mla_padded_rows():
    pitch = 576 * 2 + 16   # 1,168-byte rows
    for c in range(72 - 1):
        rows = [(lane & 15) * pitch + (c + (lane >> 4)) * 16 for lane in range(32)]
        assert _conflict_free(rows)


def test_prefill_p_stores():
    # thread r writes 16-byte chunk c of its P row (rows 32w .. 32w + 31 per warp)
    for w in range(4):
        for c in range(16):
            addrs = [_swizzled(32 * w + lane, c, 128 * 128) for lane in range(32)]
            assert _conflict_free(addrs)
