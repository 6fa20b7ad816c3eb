"""Pins of the memory / communication ledger against the values the pages print.

Every expected number comes from a fixture under tests/golden/, each citing
the page and section it was read from.
"""
import pytest

from conftest import read_golden
from oracle import ledger


def _ledger_fixture(name):
    rows = read_golden(name)
    psi = float(rows[0][1])
    n = int(rows[1][1])
    table = [r for r in rows[2:] if r[0] != "exact"]
    exact = [r for r in rows[2:] if r[0] == "exact"]
    return psi, n, table, exact


@pytest.mark.parametrize("name", ["ledger_7p5b_n64.txt", "ledger_1p5b_n8.txt"])
def test_printed_ledgers(name):
    psi, n, table, exact = _ledger_fixture(name)
    rows = ledger.ledger_rows(psi, n)
    assert len(rows) == len(table) == 4
    for row, ref in zip(rows, table):
        assert int(ref[0]) == row.stage
        assert f"{row.bytes_per_param:.4f}" == ref[1]
        assert f"{row.state_gb:.2f}" == ref[2]
        assert f"{row.saving_vs_ddp:.2f}" == ref[3]
        assert f"{row.comm_gb:.2f}" == ref[4]
    for _, stage, value in exact:
        got = ledger.gb(ledger.per_rank_state_bytes(psi, n, int(stage)))
        assert got == pytest.approx(float(value), rel=1e-12)


def test_7b_worked_table():
    rows = read_golden("ledger_7b_table.txt")
    psi = 7e9
    for r in rows:
        kind = r[0]
        if kind == "printout":
            dp = int(r[1])
            z = [ledger.gb(ledger.per_rank_state_bytes(psi, dp, s)) for s in (1, 2, 3)]
            comm = ledger.comm_elements(psi, dp, 3, exact=False) / 1e9
            assert [f"{x:.1f}" for x in z] + [f"{comm:.1f}"] == r[2:]
        elif kind == "exact":
            dp, stage, val = int(r[1]), int(r[2]), float(r[3])
            assert ledger.gb(ledger.per_rank_state_bytes(psi, dp, stage)) == pytest.approx(val,
                                                                                      rel=1e-12)
        elif kind == "table":
            dp, stage, val = int(r[1]), int(r[2]), float(r[3])
            got = ledger.gb(ledger.per_rank_state_bytes(psi, dp, stage))
            # the table rounds by hand (26.25 -> 26.3): half-up to one decimal
            assert abs(got - val) <= 0.05 + 1e-9
        elif kind == "psi70":
            dp, stage, val = int(r[1]), int(r[2]), float(r[3])
            assert ledger.gb(ledger.per_rank_state_bytes(70e9, dp, stage)) == pytest.approx(val)
        elif kind == "comm":
            mult, values, gbytes = int(r[1]), float(r[2]), float(r[3])
            stage = 1 if mult == 2 else 3
            assert ledger.comm_elements(psi, 8, stage, exact=False) == pytest.approx(values)
            assert ledger.gb(ledger.comm_bytes(psi, 8, stage)) == pytest.approx(gbytes)
        else:
            raise AssertionError(kind)


def test_misc_printed_values():
    for r in read_golden("ledger_misc.txt"):
        kind = r[0]
        if kind == "state_gb":
            psi, n, stage, val = float(r[1]), int(r[2]), int(r[3]), float(r[4])
            assert ledger.gb(ledger.per_rank_state_bytes(psi, n, stage)) == pytest.approx(val)
        elif kind == "psi_multiple":
            n, stage, mult, pct = int(r[1]), int(r[2]), float(r[3]), int(r[4])
            per = ledger.bytes_per_param(n, stage)
            assert round(per, 2) == mult
            assert round(100 * (1 - per / 16)) == pct
        elif kind == "optimizer_share":
            n, val = int(r[1]), float(r[2])
            assert ledger.KIND_BYTES["optimizer"] / n == val
        elif kind == "parts":
            psi, n, stage = float(r[1]), int(r[2]), int(r[3])
            p_gb, g_gb, o_gb, total = (float(x) for x in r[4:8])
            sharded_p = stage >= 3
            sharded_g = stage >= 2
            sharded_o = stage >= 1
            got_p = ledger.gb(ledger.KIND_BYTES["parameters"] * psi / (n if sharded_p else 1))
            got_g = ledger.gb(ledger.KIND_BYTES["gradients"] * psi / (n if sharded_g else 1))
            got_o = ledger.gb(ledger.KIND_BYTES["optimizer"] * psi / (n if sharded_o else 1))
            assert (got_p, got_g, got_o) == pytest.approx((p_gb, g_gb, o_gb))
            assert ledger.gb(ledger.per_rank_state_bytes(psi, n, stage)) == pytest.approx(total)
        else:
            raise AssertionError(kind)


def test_one_rank_all_stages_equal():
    # [L5] answer key: at dp = 1 the three stages hold the same bytes.
    psi = 1_000_000
    vals = {ledger.per_rank_state_bytes(psi, 1, s) for s in (0, 1, 2, 3)}
    assert vals == {16 * psi}


def test_limits_and_monotonicity():
    # [DZ] section 3.3: stage 1 tends to 4 Psi (4x), stage 2 to 2 Psi (8x),
    # stage 3 is exactly 16 Psi / N.
    big = 1 << 40
    assert ledger.bytes_per_param(big, 1) == pytest.approx(4.0)
    assert ledger.bytes_per_param(big, 2) == pytest.approx(2.0)
    for n in (1, 2, 8, 64, 512):
        assert ledger.bytes_per_param(n, 3) == 16.0 / n
        m = [ledger.bytes_per_param(n, s) for s in (0, 1, 2, 3)]
        assert m == sorted(m, reverse=True)


def test_fp32_accumulation_term():
    # [L5] section 2 note: +4 Psi for stage 1 (gradients unsharded), +4 Psi / N for 2 and 3.
    psi, n = 7e9, 8
    for stage, extra in ((0, 4 * psi), (1, 4 * psi), (2, 4 * psi / n), (3, 4 * psi / n)):
        d = (ledger.per_rank_state_bytes(psi, n, stage, accumulator=True)
             - ledger.per_rank_state_bytes(psi, n, stage))
        assert d == pytest.approx(extra)


def test_communication_ledger():
    # [L5] section 3: V_RS = V_AG = (N-1)/N Psi; DDP = RS + AG; ZeRO-1/2 = 2 Psi; ZeRO-3 = 3 Psi.
    psi = 7e9
    for n in (1, 2, 8, 64):
        one = ledger.collective_volume(psi, n)
        assert one == pytest.approx((n - 1) / n * psi)
        assert ledger.comm_elements(psi, n, 0) == pytest.approx(2 * one)
        assert ledger.comm_elements(psi, n, 1) == ledger.comm_elements(psi, n, 2) \
            == ledger.comm_elements(psi, n, 0)
        assert ledger.comm_elements(psi, n, 3) == pytest.approx(1.5 * ledger.comm_elements(psi, n, 1))
    # a single rank moves nothing in the exact form ([L5] table row N_d = 1) ...
    assert ledger.comm_elements(psi, 1, 3, exact=True) == 0
    # ... while the approximate 3 Psi is what the answer-key printout shows for every dp.
    assert ledger.comm_elements(psi, 1, 3, exact=False) == 3 * psi


def test_adam_scalar_count():
    for r in read_golden("adam_worked_example.txt"):
        if r[0] == "adam_scalars":
            full, per_rank = int(r[1]), int(r[2])
    assert ledger.adam_scalars_per_rank(8, 4, sharded=False) == full
    assert ledger.adam_scalars_per_rank(8, 4, sharded=True) == per_rank


def test_rejects_non_positive():
    with pytest.raises(ValueError):
        ledger.per_rank_state_bytes(0, 8, 1)
    with pytest.raises(ValueError):
        ledger.per_rank_state_bytes(10, 0, 1)
    with pytest.raises(ValueError):
        ledger.per_rank_state_bytes(10, 8, 4)
