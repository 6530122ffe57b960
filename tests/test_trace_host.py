"""The trace reader's summary on the host (CPU): which marks count and the
times it reports, on hand-made arrays of %globaltimer values."""
import numpy as np

from combine_ep_get_layout_gb300 import trace


def _arrays():
    S = trace.SLOTS
    lay = np.zeros((8, S), np.int64)
    disp = np.zeros((8, S), np.int64)
    comb = np.zeros((8, S), np.int64)
    # the combine: 4 blocks ran, the last reducer finished at 100 000 ns
    for b in range(4):
        comb[b, [0, 1, 2, 3, 4, 5]] = [10_000, 20_000, 21_000, 24_000, 90_000, 97_000 + 1_000 * b]
        comb[b, 6] = 5 + b
    # the layout: 2 blocks; block 1 skipped "slots_written" (slot 5 holds a
    # previous launch's value, older than its entry)
    lay[0, [0, 1, 2, 3, 5]] = [95_000, 101_000, 102_000, 103_000, 104_000]
    lay[1, [0, 1, 2, 3, 5]] = [95_500, 101_000, 102_500, 103_500, 50_000]
    # the dispatch: 3 blocks, the storer's wait ends at 105 000 ns
    for b in range(3):
        disp[b, [0, 3, 1, 2, 4, 5, 7]] = [98_000, 105_000, 106_000 + 500 * b, 106_500 + 500 * b,
                                          160_000 + 1_000 * b, 160_500 + 1_000 * b, 108_000]
        disp[b, 6] = 10 + b
    return {"layout": lay, "dispatch": disp, "combine": comb}


def test_times_are_after_the_last_reducer_and_counts_are_blocks_that_ran():
    r = trace.summarize(_arrays())
    assert (r["layout"]["blocks"], r["dispatch"]["blocks"], r["combine"]["blocks"]) == (2, 3, 4)
    assert r["combine"]["reducers_done"][4] == 0.0          # t0 is the last reducer's end
    assert r["combine"]["reducers_done"][0] == -3.0
    assert r["layout"]["wait_done"] == [1.0] * 5
    assert r["dispatch"]["storer_wait_done"] == [5.0] * 5
    assert r["dispatch"]["storer_ready"][0] == 6.0 and r["dispatch"]["storer_ready"][4] == 7.0
    assert r["dispatch"]["tokens_per_block"] == [10, 10.2, 11, 11.8, 12]
    assert r["combine"]["draws_per_block"][0] == 5 and r["combine"]["draws_per_block"][4] == 8


def test_a_mark_older_than_its_blocks_entry_is_left_out():
    r = trace.summarize(_arrays())
    # only block 0 reached slots_written in the last launch
    assert r["layout"]["slots_written"] == [4.0] * 5
    a = _arrays()
    a["layout"][0, 5] = 10                                  # no block reached it
    assert trace.summarize(a)["layout"]["slots_written"] is None
