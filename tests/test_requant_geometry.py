"""Contract of the requantisation's launch geometry (host only, no GPU).

The geometry of "W4AFP8 requant ..." (sglang PR #35760, requant_launch_geometry
and its CPU tests) is tuned in bytes per lane and sized from the dispatcher's
row estimate, rounded down to a power of two so that the estimate's own
round-up ((rows + E) // E) does not double the grid; any geometry writes the
same bytes.  moe_requant_launch_geometry follows the same rules for one warp
per row and 16-byte lanes; these tests hold it to them.
"""
import pytest

SMS = 152


@pytest.fixture(scope="module")
def geo():
    from weight_only_bit_moe_gb300 import build, binding
    build.build()
    return binding.moe_requant_launch_geometry


def test_grid_bounded_by_the_machine(geo):
    for rows in (-1, 0, 1, 8, 33, 1024, 1 << 20):
        for E in (1, 8, 56, 256, 1024):
            c, t = geo(E, 7168, rows, SMS)
            assert 1 <= c <= 8 * SMS and t == 256


def test_unknown_rows_take_the_whole_machine(geo):
    for E in (8, 256):
        assert geo(E, 7168, -1, SMS)[0] == 8 * SMS
        assert geo(E, 7168, 0, SMS)[0] == 8 * SMS


def test_grid_monotone_in_the_estimate(geo):
    for E in (8, 40, 56, 128, 256):
        prev = 0
        for rows in range(1, 300):
            c = geo(E, 7168, rows, SMS)[0]
            assert c >= prev
            prev = c


def test_estimate_rounded_up_does_not_grow_the_grid(geo):
    # an exact average of `rows` (a power of two from 2 up) reported as rows + 1 keeps the grid
    for E in (8, 56, 256):
        for rows in (2, 4, 8, 16, 32, 64):
            assert geo(E, 7168, rows + 1, SMS)[0] == geo(E, 7168, rows, SMS)[0]


def test_one_warp_per_estimated_row(geo):
    # 256 experts of one row: 256 rows, 8 rows (warps) per CTA
    assert geo(256, 7168, 1, SMS)[0] == 32
    assert geo(8, 7168, 1, SMS)[0] == 1
    assert geo(40, 7168, 16, SMS)[0] == 40 * 16 // 8


def test_geometry_does_not_depend_on_width(geo):
    # lanes always move 16 bytes; K changes the work per row, not the grid
    for K in (128, 896, 3584, 7168, 16384):
        assert geo(56, K, 32, SMS) == geo(56, 7168, 32, SMS)


def test_rejects_bad_arguments(geo):
    from weight_only_bit_moe_gb300 import binding
    for args in ((0, 7168, 1, SMS), (8, 0, 1, SMS), (8, 7168, 1, 0)):
        with pytest.raises(binding.MoeError):
            geo(*args)
