"""The per-parameter Shard(0) split the pages print, for the oracle and for
the library's host layout function (no GPU needed)."""
import pytest

from conftest import read_golden

import fsdp_sharded_mixed_flatten_gb300 as zf


def _rows():
    return [(int(r[1]), int(r[2]), int(r[3]), [int(x) for x in r[4:]])
            for r in read_golden("fsdp2_2d_mesh.txt") if r[0] == "shard0"]


@pytest.mark.parametrize("dim0,row,n,expect", _rows())
def test_oracle_shard_rows_match_the_pages(oracle, dim0, row, n, expect):
    got = []
    for r in range(n):
        b, e = oracle.param_shard_bounds(dim0, row, n, r)
        got.append((e - b) // row)
    assert got == expect


@pytest.fixture(scope="module")
def lib():
    from fsdp_sharded_mixed_flatten_gb300 import build
    build.build()
    return zf.load()


@pytest.mark.parametrize("dim0,row,n,expect", _rows())
def test_library_layout_matches_the_pages(lib, dim0, row, n, expect):
    L = zf.zero_param_layout(dim0, row, n)
    assert L.numel == dim0 * row and L.shard_numel == expect[0] * row
    assert [zf.zero_shard_numel(L, r) // row for r in range(n)] == expect
