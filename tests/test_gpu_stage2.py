"""ZeRO stage 2 on one GPU: zero_reduce_grads (the mean over the Nd
replicas' slices of the shard, fused with pass 1) against the oracle's
reduction and pass 1, and a whole stage-2 step (reduction, decision, AdamW)
against the oracle's."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import (bound_of, TORCH, assert_f32, assert_lp, hp_pair, oracle_step, to_dev,  # noqa: E402
                        to_host)


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


@pytest.mark.parametrize("dtype,out_dtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", "f32"),
                                             ("f16", "f32"), ("bf16", "f16")])
@pytest.mark.parametrize("nr", [1, 2, 3, 8, 16, 17])
@pytest.mark.parametrize("n", [9, 65_541, 1_000_003])
def test_reduce_matches_oracle(zp, dtype, out_dtype, nr, n):
    scale = 256.0 if dtype == "f16" else 1.0
    reps = [zs.host_grad(n, 60 + k, 0, scale, dtype) for k in range(nr)]
    want = oracle.reduce_mean(reps, dtype, out_dtype)
    sumsq, bad = oracle.norm_overflow([want if out_dtype != "f16" else want.view(np.float16)],
                                      out_dtype, scale)
    out = torch.empty(n, dtype=TORCH[out_dtype], device="cuda")
    st = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    zp.zero_reduce_grads([to_dev(r, dtype) for r in reps], out, st, ws)
    got = to_host(out)
    assert got.tobytes() == want.tobytes(), "reduced gradient differs from the oracle"
    s = zp.parse_state(st)
    assert s["found_inf"] == float(bad) and abs(s["sumsq"] - sumsq) <= 1e-6 * sumsq


def test_reduce_overflow_and_accumulate(zp):
    n = 100_005
    reps = [zs.host_grad(n, 70 + k, 0, 1024.0, "f16") for k in range(4)]
    reps[2][n - 1] = np.inf  # the tail element of one replica
    out = torch.empty(n, dtype=torch.float16, device="cuda")
    st = zp.new_state(1024.0)
    ws = zp.new_workspace(1, n)
    zp.zero_reduce_grads([to_dev(r, "f16") for r in reps], out, st, ws)
    assert zp.parse_state(st)["found_inf"] == 1.0
    assert np.isinf(to_host(out).view(np.float16)[n - 1])
    # accumulate folds a second shard into the same global sum
    reps2 = [zs.host_grad(n, 80 + k, 0, 1024.0, "f16") for k in range(4)]
    st2 = zp.new_state(1024.0)
    zp.zero_reduce_grads([to_dev(r, "f16") for r in reps2], out, st2, ws)
    first = zp.parse_state(st2)["sumsq"]
    zp.zero_reduce_grads([to_dev(r, "f16") for r in reps2], out, st2, ws, accumulate=True)
    assert zp.parse_state(st2)["sumsq"] == 2 * first


@pytest.mark.parametrize("max_norm", [0.0, 0.5])
def test_stage2_step_against_oracle(zp, max_norm):
    """Nd = 16 replicas of a shard, reduced with pass 1 fused, then the
    decision and AdamW; three steps, every element against the oracle."""
    n, nr, scale = 1_000_003, 16, 65536.0
    ohp, ghp = hp_pair(max_norm=max_norm)
    p0 = zs.host_master(n, 90)
    dp = torch.from_numpy(p0.copy()).cuda()
    dm, dv = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    dlp = torch.zeros(n, dtype=torch.float16, device="cuda")
    dg = torch.empty(n, dtype=torch.float16, device="cuda")
    st, ws = zp.new_state(scale), zp.new_workspace(1, n)
    p, m, v, plp = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    sc = oracle.Scaler(loss_scale=scale)
    for k in range(3):
        reps = [zs.host_grad(n, 90 + k, r, sc.loss_scale, "f16") for r in range(nr)]
        zp.zero_reduce_grads([to_dev(r, "f16") for r in reps], dg, st, ws)
        zp.zero_adam_step(dg, dp, dm, dv, dlp, ghp, st, ws)
        g = oracle.reduce_mean(reps, "f16", "f16").view(np.float16)
        assert to_host(dg).tobytes() == g.view(np.uint16).tobytes()
        ost = oracle_step([g], "f16", [p], [m], [v], [plp], "f16", ohp, sc, zp.parse_state(st))
        assert_f32(dp.cpu().numpy(), p, f"master step {k}", ost.exact, bound_of(ost, "p", 0))
        assert_f32(dm.cpu().numpy(), m, f"m step {k}", ost.exact, bound_of(ost, "m", 0))
        assert_f32(dv.cpu().numpy(), v, f"v step {k}", ost.exact, bound_of(ost, "v", 0))
        assert_lp(to_host(dlp), p, "f16", f"p_lp step {k}", ost.exact, bound_of(ost, "p", 0))


@pytest.mark.parametrize("inf_at", [None, 13_000_017])
def test_reduce_across_block_groups(zp, inf_at):
    """20,000,003 elements over 16 replicas: 4,883 blocks, five groups of the
    one-shot finish (the last one partial), every element and the global
    sum of squares against the oracle; an inf in one replica inside the
    third group reaches the flag through the group finish."""
    n, nr, scale = 20_000_003, 16, 256.0
    reps = [zs.host_grad(n, 90 + k, 0, scale, "f16") for k in range(nr)]
    if inf_at is not None:
        reps[5][inf_at] = np.float16(np.inf)
    want = oracle.reduce_mean(reps, "f16", "f16")
    sumsq, bad = oracle.norm_overflow([want.view(np.float16)], "f16", scale)
    out = torch.empty(n, dtype=torch.float16, device="cuda")
    st = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    zp.zero_reduce_grads([to_dev(r, "f16") for r in reps], out, st, ws)
    got = to_host(out)
    assert got.tobytes() == want.tobytes(), "reduced gradient differs from the oracle"
    s = zp.parse_state(st)
    assert s["found_inf"] == float(bad) == (0.0 if inf_at is None else 1.0)
    if inf_at is None:
        assert abs(s["sumsq"] - sumsq) <= 1e-6 * sumsq


def test_stage2_reduce_full_size_sampled(zp):
    """The benchmark's stage-2 reduction as it is timed: the GPT-2 1.5B
    Nd=16 rank-0 shard (97,350,784 elements), 16 fp16 replicas drawn on the
    device, 23,768 blocks in 24 groups of the one-shot finish.  Sampled
    elements of the mean against the oracle, and the global sum of squares
    of the whole stored result against the oracle's pass 1 over it."""
    w = zs.WORKLOADS["gpt2_1p5b_nd16"]
    S = zp.zero_partition_layout(w["numel"](), w["nd"], w["align"]).shard_numel
    nr, scale = 16, 65536.0
    reps = []
    for r in range(nr):
        t = torch.empty(S, dtype=torch.float16, device="cuda")
        zs.device_grad_into(t, 2000 + r, 0, scale)
        reps.append(t)
    out = torch.empty(S, dtype=torch.float16, device="cuda")
    st = zp.new_state(scale)
    ws = zp.new_workspace(1, S)
    zp.zero_reduce_grads(reps, out, st, ws)
    torch.cuda.synchronize()
    idx = zs.sample_indices(S, 200_000, 21)
    ti = torch.from_numpy(idx).cuda()
    want = oracle.reduce_mean([to_host(r[ti]).view(np.float16) for r in reps], "f16", "f16")
    assert to_host(out[ti]).tobytes() == want.tobytes(), "sampled mean differs from the oracle"
    full = to_host(out).view(np.float16)
    sumsq, bad = oracle.norm_overflow([full], "f16", scale)
    s = zp.parse_state(st)
    assert s["found_inf"] == float(bad) == 0.0
    assert abs(s["sumsq"] - sumsq) <= 1e-6 * sumsq
    del reps
    torch.cuda.empty_cache()
