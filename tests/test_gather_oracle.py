"""Pins for the oracle's stage-3 pieces (CPU only): the inverse layout
(shards back to tensors and tensors into shards), the per-layer gather
schedule and the communication arithmetic.  Each is checked against
something other than itself: the fragment table of the partition (pinned on
its own by a hand-worked case), element-by-element brute force, hand-worked
values and the pages' printed ratio; planted mistakes must fail a pin."""
import inspect
import json
import os

import numpy as np
import pytest

import oracle
import zero_synth as zs


def _tensors(numel, dtype=np.float32, seed=0):
    # distinct, nonzero values, so that a misplaced element always shows
    out, base = [], 1
    for n in numel:
        out.append(np.arange(base, base + n, dtype=np.float64).astype(dtype))
        base += n
    return out


def _random_numel(rng, k, hi):
    return [int(x) for x in rng.integers(0, hi, size=k)]


# ---------------------------------------------------------------- inverse layout

@pytest.mark.parametrize("case", range(12))
def test_scatter_places_every_element_by_the_fragment_table(case):
    rng = np.random.default_rng(100 + case)
    numel = _random_numel(rng, int(rng.integers(1, 9)), 40)
    nd, align = int(rng.integers(1, 6)), int(2 ** rng.integers(0, 4))
    lay = oracle.partition_layout(numel, nd, align)
    ts = _tensors(numel)
    shards = oracle.scatter_params(ts, lay.tensor_offset, nd, lay.shard_numel)
    assert len(shards) == nd and all(s.size == lay.shard_numel for s in shards)
    covered = [np.zeros(lay.shard_numel, bool) for _ in range(nd)]
    for (t, to, r, so, ln) in lay.frags:
        for j in range(ln):
            assert shards[r][so + j] == ts[t][to + j]
            covered[r][so + j] = True
    # everything the fragments do not cover is padding, and stays zero
    for r in range(nd):
        assert not shards[r][~covered[r]].any()
    # and the gather inverts it
    back = oracle.gather_params(shards, lay.tensor_offset, numel)
    for a, b in zip(back, ts):
        assert a.dtype == b.dtype and np.array_equal(a, b)


def test_gather_element_by_element():
    # tensors of 5, 3 and 10 over Nd = 4, align 2 (S = 6): the shards hold
    # the flat positions 0..23 as values; tensor 1 must come back as flat
    # positions 5, 6, 7 -- its first element from rank 0, the rest from rank 1
    shards = [np.arange(6 * r, 6 * r + 6, dtype=np.float32) for r in range(4)]
    out = oracle.gather_params(shards, [0, 5, 8], [5, 3, 10])
    assert out[0].tolist() == [0, 1, 2, 3, 4]
    assert out[1].tolist() == [5, 6, 7]
    assert out[2].tolist() == list(range(8, 18))


def test_gather_keeps_bit_patterns():
    # NaN payloads, signed zeros and infinities move unchanged (a copy, not
    # arithmetic)
    bits = np.array([0x7E01, 0xFC00, 0x8000, 0x0001, 0x7C00, 0xFFFF], np.uint16)
    shards = [bits[:3].copy(), bits[3:].copy()]
    out = oracle.gather_params(shards, [0, 2], [2, 4])
    assert np.concatenate(out).tobytes() == bits.tobytes()


# ---------------------------------------------------------------- per-layer schedule

def test_hand_worked_plan():
    # tensors of 5, 3, 7, 1 in two layers {0, 1} and {2, 3}, Nd = 3, align 2:
    # total 16, S = ceil(16 / 6) * 2 = 6
    #   layer 0 = flat [0, 8):  rank 0 gives [0, 6) -> layer [0, 6)
    #                           rank 1 gives [6, 8) = its shard [0, 2) -> layer [6, 8)
    #   layer 1 = flat [8, 16): rank 1 gives [8, 12) = shard [2, 6) -> layer [0, 4)
    #                           rank 2 gives [12, 16) = shard [0, 4) -> layer [4, 8)
    plan = oracle.gather_plan([5, 3, 7, 1], [0, 2, 4], 3, 2)
    assert [(p.begin, p.end) for p in plan] == [(0, 8), (8, 16)]
    assert plan[0].pieces == [(0, 0, 6, 0), (1, 0, 2, 6)]
    assert plan[1].pieces == [(1, 2, 4, 0), (2, 0, 4, 4)]


@pytest.mark.parametrize("case", range(10))
def test_plan_against_brute_force(case):
    rng = np.random.default_rng(200 + case)
    numel = _random_numel(rng, int(rng.integers(1, 12)), 30)
    nd, align = int(rng.integers(1, 7)), int(2 ** rng.integers(0, 3))
    cuts = sorted(set(int(x) for x in rng.integers(0, len(numel) + 1, size=3)))
    layer_first = sorted(set([0, len(numel)] + cuts))
    plan = oracle.gather_plan(numel, layer_first, nd, align)
    S = -(-sum(numel) // (nd * align)) * align
    pos = 0
    offs = []
    for n in numel:
        offs.append(pos)
        pos += n
    offs.append(pos)
    for L, lg in enumerate(plan):
        a, b = layer_first[L], layer_first[L + 1]
        # element by element: layer position k holds flat element begin + k,
        # found in rank (begin + k) // S at shard position (begin + k) % S
        want = {}
        for t in range(a, b):
            for j in range(numel[t]):
                f = offs[t] + j
                want[f - offs[a]] = (f // S, f % S)
        got = {}
        for (r, so, ln, lo) in lg.pieces:
            assert ln > 0
            for k in range(ln):
                assert lo + k not in got
                got[lo + k] = (r, so + k)
        assert got == want
        assert (lg.begin, lg.end) == (offs[a], offs[b])
        ranks = [p[0] for p in lg.pieces]
        assert ranks == sorted(set(ranks))  # one piece per rank, in rank order


def test_plan_of_the_gpt2_layers():
    numel = zs.WORKLOADS["gpt2_1p5b_nd16"]["numel"]()
    lf = zs.gpt2_layer_first()
    assert lf[0] == 0 and lf[-1] == len(numel) == 580 and len(lf) == 51
    plan = oracle.gather_plan(numel, lf, 16, 128)
    S = 97_350_784
    h = 1600
    block = 12 * h * h + 13 * h
    sizes = [lg.end - lg.begin for lg in plan]
    assert sizes[0] == (50257 + 1024) * h and sizes[-1] == 2 * h
    assert sizes[1:-1] == [block] * 48
    assert sum(sizes) == sum(numel)
    for lg in plan:
        assert sum(p[2] for p in lg.pieces) == lg.end - lg.begin
        # a block (30.8M params) is smaller than a shard, so it needs at
        # most two ranks
        if lg.end - lg.begin <= S:
            assert len(lg.pieces) <= 2


# ---------------------------------------------------------------- communication

def test_stage3_communication_matches_pages():
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "memory_pages.json")))
    extra = gold["stage_reduction"]["stage3_extra_comm"]
    psi = 1.5e9
    dp = oracle.comm_volume(psi, 0)
    assert oracle.comm_volume(psi, 1) == dp and oracle.comm_volume(psi, 2) == dp
    assert oracle.comm_volume(psi, 3) / dp - 1.0 == extra


# ---------------------------------------------------------------- the pins can fail

PINS = [
    lambda: [test_scatter_places_every_element_by_the_fragment_table(c) for c in range(12)],
    test_gather_element_by_element,
    test_gather_keeps_bit_patterns,
    test_hand_worked_plan,
    lambda: [test_plan_against_brute_force(c) for c in range(10)],
    test_plan_of_the_gpt2_layers,
    test_stage3_communication_matches_pages,
]

# (function, text in its source, replacement)
MUTANTS = [
    ("gather_params", "full[o:o + n]", "full[o + 1:o + n + 1]"),
    ("gather_params", "np.concatenate(shards)", "np.concatenate(shards[::-1])"),
    ("scatter_params", "full[r * shard_numel:(r + 1) * shard_numel]",
     "full[r * shard_numel + 1:(r + 1) * shard_numel + 1]"),
    ("gather_plan", "lo - begin", "lo - r * S"),
    ("gather_plan", "min(end, (r + 1) * S)", "min(end, r * S + S - 1)"),
    ("gather_plan", "lo - r * S, hi - lo", "lo - begin, hi - lo"),
    ("comm_volume", "return 3.0 * psi", "return 4.0 * psi"),
]


def _mutated(name, old, new):
    src = inspect.getsource(getattr(oracle, name))
    assert old in src, (name, old)
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns[name]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[f"{m[0]}:{i}" for i, m in enumerate(MUTANTS)])
def test_planted_mistake_is_caught(name, old, new, monkeypatch):
    monkeypatch.setattr(oracle, name, _mutated(name, old, new))
    failed = 0
    for pin in PINS:
        try:
            pin()
        except Exception:
            failed += 1
    assert failed > 0, f"no pin caught the mistake in {name}: {old!r} -> {new!r}"
