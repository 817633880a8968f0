"""ZeRO stage 3 on one GPU: zero_gather_params (shards -> tensors),
zero_scatter_params (tensors -> shards) and the per-layer schedule of
zero_gather_plan, against the oracle's inverse layout, bit for bit.  Element
values are random bit patterns (NaN and infinity patterns included), so any
conversion, reordering or misplaced element shows."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import TORCH, to_host  # noqa: E402

BITS = {"f16": np.uint16, "bf16": np.uint16, "f32": np.uint32}


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def rand_bits(rng, n, dtype):
    t = BITS[dtype]
    return rng.integers(0, np.iinfo(t).max, size=n, dtype=t, endpoint=True)


def to_dev_bits(a, dtype):
    """Upload a bit-pattern array as a device tensor of the element type."""
    if dtype == "f32":
        return torch.from_numpy(a.view(np.int32).copy()).view(torch.float32).cuda()
    return torch.from_numpy(a.view(np.int16).copy()).view(TORCH[dtype]).cuda()


def host_bits(t, dtype):
    return to_host(t).view(BITS[dtype])


def layouts():
    """(numel, nd, align): ragged tensors, empty ones, tensors longer than a
    16 KiB tile, shards shorter than a tile (several rank boundaries inside
    one tile) and the reverse."""
    rng = np.random.default_rng(7)
    out = [([5, 3, 10], 4, 2), ([1], 1, 1), ([0, 0, 7, 0], 3, 1), ([40_000, 12_345, 3, 70_001], 3, 128)]
    for _ in range(6):
        k = int(rng.integers(1, 30))
        numel = [int(x) for x in rng.integers(0, 20_000, k)]
        numel[int(rng.integers(0, k))] = int(rng.integers(0, 3))
        out.append((numel, int(rng.integers(1, 17)), int(2 ** rng.integers(0, 8))))
    out.append(([int(x) for x in rng.integers(1, 300, 200)], 16, 8))  # many short tensors
    # more shards than the kernel argument block holds (the table goes
    # through the workspace), with few and with many tensors
    out.append(([int(x) for x in rng.integers(0, 50, 20)], 300, 1))
    out.append(([int(x) for x in rng.integers(0, 50, 100)], 300, 2))
    return out


LAYOUTS = layouts()


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("case", range(len(LAYOUTS)))
def test_gather_matches_oracle(zp, dtype, case):
    numel, nd, align = LAYOUTS[case]
    lay = oracle.partition_layout(numel, nd, align)
    S = lay.shard_numel
    rng = np.random.default_rng(1000 + case)
    shards = [rand_bits(rng, S, dtype) for _ in range(nd)]
    want = oracle.gather_params(shards, lay.tensor_offset, numel)
    d_shards = [to_dev_bits(s, dtype) for s in shards]
    # separate allocations, pre-filled with a value the gather must overwrite
    d_tens = [torch.full((n,), 123.0, dtype=TORCH[dtype], device="cuda") for n in numel]
    ws = torch.empty(zp.zero_gather_workspace_bytes(len(numel), nd), dtype=torch.uint8, device="cuda")
    zp.zero_gather_params(d_shards, d_tens, lay.tensor_offset, ws)
    torch.cuda.synchronize()
    for i, (t, w) in enumerate(zip(d_tens, want)):
        got = host_bits(t, dtype)
        assert got.tobytes() == w.tobytes(), f"tensor {i} (numel {numel[i]}) differs"


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("case", range(len(LAYOUTS)))
def test_scatter_matches_oracle(zp, dtype, case):
    numel, nd, align = LAYOUTS[case]
    lay = oracle.partition_layout(numel, nd, align)
    S = lay.shard_numel
    rng = np.random.default_rng(2000 + case)
    tens = [rand_bits(rng, n, dtype) for n in numel]
    want = oracle.scatter_params(tens, lay.tensor_offset, nd, S) if tens else []
    sentinel = {"f16": 0x7E55, "bf16": 0x7FD5, "f32": 0x7FC05555}[dtype]
    d_shards = [to_dev_bits(np.full(S, sentinel, BITS[dtype]), dtype) for _ in range(nd)]
    d_tens = [to_dev_bits(t, dtype) for t in tens]
    ws = torch.empty(zp.zero_gather_workspace_bytes(len(numel), nd), dtype=torch.uint8, device="cuda")
    zp.zero_scatter_params(d_tens, lay.tensor_offset, d_shards, ws)
    torch.cuda.synchronize()
    total = sum(numel)
    for r in range(nd):
        got = host_bits(d_shards[r], dtype)
        flat = np.arange(r * S, (r + 1) * S)
        real = flat < total
        # tensor elements as the oracle places them; the padding untouched
        assert got[real].tobytes() == want[r][real].tobytes(), f"shard {r} differs"
        assert (got[~real] == sentinel).all(), f"shard {r}: padding was written"


def test_per_layer_gather_of_a_small_gpt(zp):
    """The stage-3 schedule: each layer gathered into one reused layer buffer
    (a one-entry list at the layer's flat offset), its tensors views of it."""
    shapes = zs.gpt2_shapes(layers=4, hidden=64, vocab=1000, positions=128)
    numel = zs.numels(shapes)
    lf = zs.gpt2_layer_first(4)
    nd = 16
    lay = oracle.partition_layout(numel, nd, 128)
    plan_ref = oracle.gather_plan(numel, lf, nd, 128)
    plan = zp.zero_gather_plan(numel, lf, nd, 128)
    rng = np.random.default_rng(5)
    shards = [rand_bits(rng, lay.shard_numel, "f16") for _ in range(nd)]
    d_shards = [to_dev_bits(s, "f16") for s in shards]
    buf = torch.empty(plan.max_layer_numel, dtype=torch.float16, device="cuda")
    ws = torch.empty(zp.zero_gather_workspace_bytes(1, nd), dtype=torch.uint8, device="cuda")
    for L, lg in enumerate(plan_ref):
        n = lg.end - lg.begin
        assert (int(plan.layer_flat[L]), int(plan.layer_flat[L + 1])) == (lg.begin, lg.end)
        view = buf[:n]
        zp.zero_gather_params(d_shards, [view], [lg.begin], ws)
        got = host_bits(view, "f16")
        # the oracle's per-layer plan: each piece from its rank's shard
        want = np.empty(n, np.uint16)
        for (r, so, ln, lo) in lg.pieces:
            want[lo:lo + ln] = shards[r][so:so + ln]
        assert got.tobytes() == want.tobytes(), f"layer {L}"
        # and the tensors of the layer are the oracle's gathered tensors
        ts = oracle.gather_params(shards, lay.tensor_offset[lf[L]:lf[L + 1]], numel[lf[L]:lf[L + 1]])
        if ts:
            assert np.concatenate(ts).tobytes() == want.tobytes()
        else:
            assert n == 0


def test_gather_full_gpt2_nd16_sampled(zp):
    """The benchmark's call at full size: the GPT-2 1.5B parameters (580
    tensors, 1,557,611,200 fp16 elements) gathered from 16 shards in one
    launch; a sample of tensors (first, last, the largest, random ones)
    compared whole with the oracle, and every tensor's ends checked."""
    numel = zs.WORKLOADS["gpt2_1p5b_nd16"]["numel"]()
    nd = 16
    lay = oracle.partition_layout(numel, nd, 128)
    S = lay.shard_numel
    rng = np.random.default_rng(11)
    shards = [rand_bits(rng, S, "f16") for _ in range(nd)]
    d_shards = [to_dev_bits(s, "f16") for s in shards]
    d_tens = [torch.empty(n, dtype=torch.float16, device="cuda") for n in numel]
    ws = torch.empty(zp.zero_gather_workspace_bytes(len(numel), nd), dtype=torch.uint8, device="cuda")
    zp.zero_gather_params(d_shards, d_tens, lay.tensor_offset, ws)
    torch.cuda.synchronize()
    pick = sorted({0, 1, 2, len(numel) - 1, len(numel) - 2, int(np.argmax(numel))} |
                  {int(x) for x in rng.integers(0, len(numel), 12)})
    want = oracle.gather_params(shards, [lay.tensor_offset[i] for i in pick], [numel[i] for i in pick])
    for i, w in zip(pick, want):
        assert host_bits(d_tens[i], "f16").tobytes() == w.tobytes(), f"tensor {i}"
    full = np.concatenate(shards)
    for i, t in enumerate(d_tens):
        o, n = lay.tensor_offset[i], numel[i]
        k = min(n, 64)
        assert host_bits(t[:k], "f16").tobytes() == full[o:o + k].tobytes(), f"tensor {i} head"
        assert host_bits(t[n - k:], "f16").tobytes() == full[o + n - k:o + n].tobytes(), f"tensor {i} tail"


def test_scatter_then_gather_round_trip_frag_sizes(zp):
    """10,000 log-normal tensors (the fragmented workload's sizes, scaled to
    a tenth) scattered into 7 shards and gathered back: the identity."""
    sizes = [max(1, n // 10) for n in zs.frag_sizes()]
    nd = 7
    lay = oracle.partition_layout(sizes, nd, 128)
    rng = np.random.default_rng(3)
    tens = [rand_bits(rng, n, "bf16") for n in sizes]
    d_tens = [to_dev_bits(t, "bf16") for t in tens]
    d_shards = [torch.zeros(lay.shard_numel, dtype=torch.bfloat16, device="cuda") for _ in range(nd)]
    ws = torch.empty(zp.zero_gather_workspace_bytes(len(sizes), nd), dtype=torch.uint8, device="cuda")
    lst = zp.TensorList(d_tens)
    zp.zero_scatter_params(lst, lay.tensor_offset, d_shards, ws)
    back = [torch.empty_like(t) for t in d_tens]
    zp.zero_gather_params(d_shards, zp.TensorList(back), lay.tensor_offset, ws)
    torch.cuda.synchronize()
    want = oracle.scatter_params(tens, lay.tensor_offset, nd, lay.shard_numel)
    for r in range(nd):
        assert host_bits(d_shards[r], "bf16").tobytes() == want[r].tobytes()
    got = torch.cat(back).cpu().view(torch.int16).numpy().view(np.uint16)
    assert got.tobytes() == np.concatenate(tens).tobytes()


def test_gather_argument_errors(zp):
    f16 = torch.float16
    shards = [torch.zeros(64, dtype=f16, device="cuda") for _ in range(2)]
    ws = torch.empty(zp.zero_gather_workspace_bytes(4, 2), dtype=torch.uint8, device="cuda")
    t = torch.empty(10, dtype=f16, device="cuda")
    with pytest.raises(zp.ZeroError) as e:   # past the flat end (128 elements)
        zp.zero_gather_params(shards, [t], [120], ws)
    assert e.value.code == -8
    big = torch.empty(16, dtype=f16, device="cuda")
    with pytest.raises(zp.ZeroError) as e:   # a view that starts 2 bytes in
        zp.zero_gather_params(shards, [big[1:9]], [0], ws)
    assert e.value.code == -2
    a, b = torch.empty(10, dtype=f16, device="cuda"), torch.empty(10, dtype=f16, device="cuda")
    with pytest.raises(zp.ZeroError) as e:   # scatter of overlapping ranges
        zp.zero_scatter_params([a, b], [0, 5], shards, ws)
    assert e.value.code == -8
    zp.zero_gather_params(shards, [a, b], [0, 5], ws)  # overlapping reads are fine
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(zp.ZeroError) as e:
        zp.zero_gather_params(shards, [t], [0], small)
    assert e.value.code == -5
    with pytest.raises(TypeError):
        zp.zero_gather_params(shards, [torch.empty(4, device="cuda")], [0], ws)
    # nothing to do: an empty list and empty tensors
    zp.zero_gather_params(shards, [], [], ws)
    zp.zero_gather_params(shards, [torch.empty(0, dtype=f16, device="cuda")], [128], ws)
    torch.cuda.synchronize()
