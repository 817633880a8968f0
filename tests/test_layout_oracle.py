"""Pins for the oracle's flat partition layout (CPU only): a hand-worked
case, the sizes of the workloads' shards, and coverage invariants."""
import numpy as np
import pytest

import oracle
import zero_synth as zs


def test_hand_worked_layout():
    # tensors of 5, 3 and 10 elements over Nd = 4 ranks, align 2:
    # total 18, S = ceil(18 / 8) * 2 = 6, padded 24
    #   flat: t0 [0,5) t1 [5,8) t2 [8,18) pad [18,24)
    #   rank 0 [0,6):  t0[0:5], t1[0:1]
    #   rank 1 [6,12): t1[1:3], t2[0:4]
    #   rank 2 [12,18): t2[4:10]
    #   rank 3 [18,24): padding only
    lay = oracle.partition_layout([5, 3, 10], 4, 2)
    assert lay.shard_numel == 6 and lay.padded_total == 24
    assert lay.tensor_offset == [0, 5, 8]
    assert lay.frags == [(0, 0, 0, 0, 5), (1, 0, 0, 5, 1), (1, 1, 1, 0, 2),
                         (2, 0, 1, 2, 4), (2, 4, 2, 0, 6)]


def test_workload_shard_sizes():
    tiny = oracle.partition_layout(zs.WORKLOADS["tiny"]["numel"](), 1, 128)
    assert sum(zs.WORKLOADS["tiny"]["numel"]()) == 1_836_288
    assert tiny.shard_numel == 1_836_288 and tiny.padded_total == 1_836_288
    g = zs.WORKLOADS["gpt2_1p5b_nd16"]["numel"]()
    assert len(g) == 580 and sum(g) == 1_557_611_200
    l16 = oracle.partition_layout(g, 16, 128)
    assert l16.shard_numel == 97_350_784
    assert l16.padded_total - sum(g) == 1_344
    l1 = oracle.partition_layout(g, 1, 128)
    assert l1.shard_numel == 1_557_611_264
    s = zs.WORKLOADS["stack_100b_nd400"]["numel"]()
    assert len(s) == 1500 and sum(s) == 100_676_608_000
    l400 = oracle.partition_layout(s, 400, 128)
    assert l400.shard_numel == 251_691_520 and l400.padded_total == sum(s)


def check_invariants(numel, nd, align):
    lay = oracle.partition_layout(numel, nd, align)
    total = sum(numel)
    S = lay.shard_numel
    assert S % align == 0 and lay.padded_total == nd * S
    assert lay.padded_total >= total and lay.padded_total - total < nd * align
    cover = np.zeros(lay.padded_total, np.int32)
    for t, toff, r, soff, ln in lay.frags:
        assert 0 <= r < nd and 0 <= soff and soff + ln <= S and ln > 0
        assert 0 <= toff and toff + ln <= numel[t]
        flat = r * S + soff
        assert flat == lay.tensor_offset[t] + toff
        cover[flat:flat + ln] += 1
    # every element of every tensor exactly once, padding only at the tail
    assert np.all(cover[:total] == 1) and not cover[total:].any()
    # fragments of one tensor tile it in order
    for t, n in enumerate(numel):
        parts = [(toff, ln) for tt, toff, _, _, ln in lay.frags if tt == t]
        pos = 0
        for toff, ln in parts:
            assert toff == pos
            pos += ln
        assert pos == n


@pytest.mark.parametrize("seed", range(20))
def test_random_layout_invariants(seed):
    rng = np.random.default_rng(seed)
    k = int(rng.integers(1, 40))
    numel = [int(x) for x in rng.integers(0, 300, k)]
    nd = int(rng.integers(1, 17))
    align = int(2 ** rng.integers(0, 6))
    check_invariants(numel, nd, align)


def test_degenerate_layouts():
    lay = oracle.partition_layout([], 4, 8)
    assert lay.shard_numel == 0 and lay.frags == []
    lay = oracle.partition_layout([0, 0], 3, 4)
    assert lay.shard_numel == 0 and lay.frags == []
    check_invariants([1], 7, 1)
    check_invariants([0, 5, 0], 2, 4)
    with pytest.raises(ValueError):
        oracle.partition_layout([3], 0, 1)
