"""Pins of the packed-transfer oracle (oracle/transfer.py)."""
import numpy as np
import pytest

import oracle
from oracle import transfer

G, L, R = 0, 1, 2


@pytest.mark.parametrize("P", [16, 64])
def test_rows_hold_everything_a_later_query_can_see(P):
    # whatever the last position (or a query right after it) may see must travel
    rng = np.random.default_rng(P)
    idx = sorted(rng.choice(5000, size=300, replace=False).tolist())
    for pol in [(G, 0, 0, None), (L, 4, 1024, None), (L, 0, 1, None), (L, 130, 64, None),
                (R, 0, 0, idx)]:
        for n in (1, 7, 300, 4096):
            rows = set(transfer.unit_rows(*pol, n, P))
            need = set(oracle.visible(pol[0], pol[1], pol[2], pol[3], n - 1).tolist())
            assert need <= rows, (pol, n)
            assert all(0 <= r < n for r in rows)


def test_row_sets_by_class():
    assert transfer.unit_rows(G, 0, 0, None, 10, 16) == list(range(10))
    idx = [3, 8, 9, 40]
    assert transfer.unit_rows(R, 0, 0, idx, 20, 16) == [3, 8, 9]
    # LOCAL(4, 40) at P = 16 keeps the sink and a ring of ceil(40/16)+1 = 4 pages
    rows = transfer.unit_rows(L, 4, 40, None, 1000, 16)
    assert rows == list(range(4)) + list(range(1000 - 64, 1000))


def test_transfer_ratio_closed_form():
    # one LOCAL(4, 2048) head at P = 64 over 32,768 tokens: dense / kept =
    # 32768 / (4 + 33 * 64)
    pol = [[(L, 4, 2048, None)]]
    assert transfer.transfer_ratio(pol, [32768], 64) == pytest.approx(32768 / (4 + 33 * 64))
    # GLOBAL keeps everything
    assert transfer.transfer_ratio([[(G, 0, 0, None)]], [777], 64) == 1.0


def test_payload_order():
    n, d = 50, 2
    k = np.arange(n * 1 * d, dtype=np.float64).reshape(n, 1, d)
    v = -k
    pol = [[(R, 0, 0, [5, 7, 49])]]
    got = transfer.payload(pol, [n], [k], [v], 16)
    want = np.concatenate([k[[5, 7, 49], 0].reshape(-1), v[[5, 7, 49], 0].reshape(-1)])
    np.testing.assert_array_equal(got, want)
