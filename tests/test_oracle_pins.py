"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
import _pins


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(o, pin):
    pin(o)


def test_brute_force_n10_worked_example_unique(o):
    pts, perm, _ = _pins.load_worked_example()
    cnt, first = o.brute_force(pts, mode=1)
    assert cnt == 1
    assert (o.build_tree(pts, mode=1) == first).all()


def test_balanced_brute_force_n10_unique(o):
    pts, _, _ = _pins.load_worked_example()
    for p in (pts, pts[:, ::-1].copy()):
        cnt, first = o.brute_force_balanced(p)
        assert cnt == 1
        assert (o.build_balanced(p) == first).all()


def test_oracle_rejects_bad_input(o):
    import numpy as np
    pts = np.zeros((4, 2), dtype=np.float32)
    pts[2, 1] = np.nan
    with pytest.raises(oracle.OracleError) as e:
        o.build_tree(pts)
    assert e.value.code == oracle.ENONFINITE
    pts[2, 1] = np.inf
    with pytest.raises(oracle.OracleError):
        o.build_tree(pts)
    with pytest.raises(oracle.OracleError):
        o.build_tree(np.zeros((0, 3), dtype=np.float32))
    with pytest.raises(oracle.OracleError):
        o.build_tree(np.zeros((3, 3), dtype=np.float32), mode=2)


def test_small_edge_sizes(o):
    import numpy as np
    assert list(o.build_tree(np.array([[3.0]], dtype=np.float32))) == [0]
    # N=2: the root takes rank |S(1)| = 1, i.e. the larger point; node 1 the smaller
    assert list(o.build_tree(np.array([[2.0], [1.0]], dtype=np.float32))) == [0, 1]
    assert list(o.build_tree(np.array([[1.0], [2.0]], dtype=np.float32))) == [1, 0]
    # equal points: the index breaks the tie
    assert list(o.build_tree(np.array([[1.0], [1.0]], dtype=np.float32))) == [1, 0]
