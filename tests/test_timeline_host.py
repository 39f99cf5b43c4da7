"""Host logic of the decode timeline tool: each stamp relative to the
previous launch's last exit, median and latest over CTAs, and stamps a
kernel shape never passes shown as absent."""
import numpy as np

from kv_cache_eviction_03_gb300 import timeline as T


def launch(base, grid, rng, skip=()):
    st = np.zeros((grid, T.NSTAMP), dtype=np.int64)
    for k, (_, i) in enumerate(T.STAMPS):
        if i in skip:
            continue
        st[:, i] = base + 1000 * k + rng.integers(0, 100, size=grid)
    return st


def test_phase_table_is_relative_to_previous_exit():
    rng = np.random.default_rng(0)
    grid = 9
    launches = [launch(b, grid, rng) for b in (0, 20_000, 40_000)]
    rows = T.phase_table(launches)
    assert len(rows) == 2
    for prev, cur, row in zip(launches[:-1], launches[1:], rows):
        end = prev[:, T.EXIT].max()
        for name, i in T.STAMPS:
            med, latest = row[name]
            assert np.isclose(med, np.median(cur[:, i] - end) / 1e3)
            assert np.isclose(latest, (cur[:, i].max() - end) / 1e3)


def test_unwritten_stamp_is_absent():
    rng = np.random.default_rng(1)
    pushed = dict(T.STAMPS)["candidate pushed"]
    launches = [launch(b, 4, rng, skip=(pushed,)) for b in (0, 20_000)]
    row = T.phase_table(launches)[0]
    assert row["candidate pushed"] is None
    assert row["exit"] is not None and row["victim known"][0] < row["exit"][0]


def test_stamp_order_and_indices():
    names = [n for n, _ in T.STAMPS]
    idx = [i for _, i in T.STAMPS]
    assert names[0] == "entry" and names[-1] == "exit" and dict(T.STAMPS)["exit"] == T.EXIT
    assert sorted(idx) == list(range(T.NSTAMP))
