"""GPU parity: the CUDA path through the C ABI against the oracle, element by
element, on the seeded synthetic workloads (their full sizes, with sampled
elements where the host cannot update the whole shard) and on ragged and
degenerate sizes.  See gpu_common for the bar."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import (bound_of, TORCH, assert_f32, assert_lp, assert_lp_copy, hp_pair, oracle_step, to_dev,  # noqa: E402
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


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def run_full(zp, n, gdtype, pdtype, steps, scale, max_norm=0.0, seed=0, inf_step=None,
             inf_pos=None, nan=False, hp_kw=None, whole=False):
    """Full-array comparison of a flat shard of n elements over `steps` steps
    (whole: the step through zero_step, else pass 1 and zero_adam_step)."""
    ohp, ghp = hp_pair(max_norm=max_norm, **(hp_kw or {}))
    p0 = zs.host_master(n, seed)
    dp = torch.from_numpy(p0.copy()).cuda()
    dm = torch.zeros(n, dtype=torch.float32, device="cuda")
    dv = torch.zeros(n, dtype=torch.float32, device="cuda")
    dlp = torch.zeros(n, dtype=TORCH[pdtype], device="cuda")
    state = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    plp = np.zeros(n, np.uint16)
    sc = oracle.Scaler(loss_scale=scale)
    skipped = 0
    for k in range(steps):
        g = zs.host_grad(n, seed, k, sc.loss_scale, gdtype)
        if inf_step == k and n > 0:
            pos = zs.inf_index(n, seed, k) if inf_pos is None else inf_pos
            bad = np.float32(np.nan if nan else np.inf)
            g[pos] = zs.host_cast(np.array([bad], np.float32), gdtype)[0]
        dg = to_dev(g, gdtype)
        before = [to_host(t) for t in (dp, dm, dv, dlp)]
        if whole:
            zp.zero_step(dg, dp, dm, dv, dlp, ghp, state, ws)
        else:
            zp.zero_grad_norm_overflow(dg, state, ws)
            zp.zero_adam_step(dg, dp, dm, dv, dlp, ghp, state, ws)
        gst = zp.parse_state(state)
        st = oracle_step([g], gdtype, [p], [m], [v], [plp], pdtype, ohp, sc, gst)
        after = [to_host(t) for t in (dp, dm, dv, dlp)]
        if st.skip:
            skipped += 1
            for a, b in zip(after, before):
                assert a.tobytes() == b.tobytes(), "a skipped step changed the state"
        assert_f32(after[0], p, f"master step {k}", st.exact, bound_of(st, "p", 0))
        assert_f32(after[1], m, f"m step {k}", st.exact, bound_of(st, "m", 0))
        assert_f32(after[2], v, f"v step {k}", st.exact, bound_of(st, "v", 0))
        assert_lp_copy(after[3], plp, f"p_lp step {k} against the oracle's copy", st.exact)
        if skipped < k + 1:  # at least one step applied: p_lp is the rounded master
            assert_lp(after[3], p, pdtype, f"p_lp step {k}", st.exact, bound_of(st, "p", 0))
    return zp.parse_state(state), skipped


# ------------------------------------------------------------------ workloads

def test_tiny_transformer(zp):
    """The 2-layer, hidden-256 transformer state (14 tensors, Nd = 1),
    fp16 grads x 1024, 3 steps: every element of every step."""
    w = zs.WORKLOADS["tiny"]
    lay = zp.zero_partition_layout(w["numel"](), w["nd"], w["align"])
    st, skipped = run_full(zp, lay.shard_numel, "f16", "f16", w["steps"], w["loss_scale"])
    assert st["step"] == 3 and skipped == 0


def test_gpt2_nd16_shard_with_overflow(zp):
    """GPT-2 1.5B flattened into 16 shards: rank 0's 97,350,784-element shard,
    fp16 grads x 65536, one +inf at a seeded index in step 2 (index 1 of 5):
    that step is skipped with the state byte-identical and the scale halved;
    every element of every step compared.  This is also the launch
    configuration the benchmark times."""
    w = zs.WORKLOADS["gpt2_1p5b_nd16"]
    lay = zp.zero_partition_layout(w["numel"](), w["nd"], w["align"])
    assert lay.shard_numel == 97_350_784
    st, skipped = run_full(zp, lay.shard_numel, "f16", "f16", w["steps"], w["loss_scale"],
                           inf_step=1)
    assert skipped == 1 and st["skipped"] == 1 and st["step"] == 4
    assert st["loss_scale"] == 32768.0


def sampled_run(zp, n, gdtype, pdtype, steps, scale, max_norm, micro=1, seed=0, count=200_000):
    """Full-size run on the GPU with device-drawn inputs; the oracle computes
    the global norm over the whole gradient (copied to the host) and follows
    a sample of elements through every step."""
    ohp, ghp = hp_pair(max_norm=max_norm)
    dp = torch.empty(n, dtype=torch.float32, device="cuda")
    zs.device_master_into(dp, seed)
    idx = zs.sample_indices(n, count, seed)
    didx = torch.from_numpy(idx).cuda()
    p = dp[didx].cpu().numpy()
    m = np.zeros(idx.size, np.float32)
    v = np.zeros(idx.size, np.float32)
    plp = np.zeros(idx.size, np.uint16)
    dm = torch.zeros(n, dtype=torch.float32, device="cuda")
    dv = torch.zeros(n, dtype=torch.float32, device="cuda")
    dlp = torch.zeros(n, dtype=TORCH[pdtype], device="cuda")
    state = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    sc = oracle.Scaler(loss_scale=scale)
    acc = torch.empty(n, dtype=torch.float32, device="cuda") if micro > 1 else None
    for k in range(steps):
        if micro > 1:
            bufs = [torch.empty(n, dtype=TORCH[gdtype], device="cuda") for _ in range(micro)]
            for j, b in enumerate(bufs):
                zs.device_grad_into(b, seed, k, sc.loss_scale, micro=j)
            zp.zero_accumulate_grads(acc, bufs, overwrite=True)
            host_bufs = [to_host(b) for b in bufs]
            del bufs
            g_host = np.empty(n, np.float32)
            oracle.accumulate(g_host, host_bufs, gdtype, overwrite=True)
            del host_bufs
            got = acc.cpu().numpy()
            assert got.tobytes() == g_host.tobytes(), "accumulated gradient differs"
            del got
            dg, g_dtype = acc, "f32"
        else:
            dg = torch.empty(n, dtype=TORCH[gdtype], device="cuda")
            zs.device_grad_into(dg, seed, k, sc.loss_scale)
            g_host = to_host(dg)
            g_dtype = gdtype
        zp.zero_grad_norm_overflow(dg, state, ws)
        zp.zero_adam_step(dg, dp, dm, dv, dlp, ghp, state, ws)
        gst = zp.parse_state(state)
        st = oracle_step([g_host], g_dtype, [p], [m], [v], [plp], pdtype, ohp, sc, gst,
                         sampled_idx=idx)
        del g_host
        assert_f32(dp[didx].cpu().numpy(), p, f"master step {k}", st.exact, bound_of(st, "p", 0))
        assert_f32(dm[didx].cpu().numpy(), m, f"m step {k}", st.exact, bound_of(st, "m", 0))
        assert_f32(dv[didx].cpu().numpy(), v, f"v step {k}", st.exact, bound_of(st, "v", 0))
        assert_lp(to_host(dlp[didx]), p, pdtype, f"p_lp step {k}", st.exact, bound_of(st, "p", 0))
    return zp.parse_state(state)


def test_gpt2_full_unpartitioned_clip(zp):
    """The whole 1.5B-param state on one GPU (Nd = 1, 1,557,611,264 elements
    after padding), fp16 grads, global-norm clip 1.0, 3 steps."""
    w = zs.WORKLOADS["gpt2_1p5b_full"]
    lay = zp.zero_partition_layout(w["numel"](), w["nd"], w["align"])
    st = sampled_run(zp, lay.shard_numel, "f16", "f16", w["steps"], w["loss_scale"], w["max_norm"])
    assert st["step"] == 3 and st["last_clip"] < 1.0  # norm ~ 39.5: clipping active


def test_100b_nd400_shard_accumulate_clip(zp):
    """Rank 0's 251,691,520-element shard of the 100B layer stack over 400
    ranks: 4 bf16 micro-batch gradients accumulated into fp32, clip 1.0 over
    the shard, bf16 parameters, 3 steps."""
    w = zs.WORKLOADS["stack_100b_nd400"]
    lay = zp.zero_partition_layout(w["numel"](), w["nd"], w["align"])
    assert lay.shard_numel == 251_691_520
    st = sampled_run(zp, lay.shard_numel, "bf16", "bf16", w["steps"], w["loss_scale"],
                     w["max_norm"], micro=w["micro_batches"])
    assert st["step"] == 3 and st["last_clip"] < 1.0


@pytest.mark.parametrize("k", [16, 20, 24])
def test_sweep_flat_full(zp, k):
    """Flat shards of 2^k elements (and 2^k + 3, a ragged tail), fp16."""
    for n in (1 << k, (1 << k) + 3):
        run_full(zp, n, "f16", "f16", 3, 1024.0)


def test_sweep_flat_2pow31_sampled(zp):
    """A shard of 2^31 + 5 elements: 64-bit indexing, ragged tail; the sample
    includes the last 4096 elements, past index 2^31."""
    n = (1 << 31) + 5
    st = sampled_run(zp, n, "f16", "f16", 2, 1024.0, 0.0, count=50_000)
    assert st["step"] == 2


def test_frag_10k_list(zp):
    """The 10,000-tensor list with log-normal sizes (median 4096, max 2^24),
    each tensor its own allocation, updated through the multi-tensor path;
    every element of every tensor compared over 3 steps."""
    w = zs.WORKLOADS["frag_10k"]
    sizes = w["numel"]()
    scale = w["loss_scale"]
    ohp, ghp = hp_pair()
    total = sum(sizes)
    p0 = zs.host_master(total, 0)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    hp_ = [p0[offs[i]:offs[i + 1]].copy() for i in range(len(sizes))]
    hm = [np.zeros(s, np.float32) for s in sizes]
    hv = [np.zeros(s, np.float32) for s in sizes]
    hl = [np.zeros(s, np.uint16) for s in sizes]
    dp = [torch.from_numpy(a.copy()).cuda() for a in hp_]
    dm = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in sizes]
    dv = [torch.zeros(s, dtype=torch.float32, device="cuda") for s in sizes]
    dl = [torch.zeros(s, dtype=torch.float16, device="cuda") for s in sizes]
    state = zp.new_state(scale)
    ws = zp.new_workspace(len(sizes), total)
    sc = oracle.Scaler(loss_scale=scale)
    for k in range(w["steps"]):
        gflat = zs.host_grad(total, 0, k, sc.loss_scale, "f16")
        gl = [gflat[offs[i]:offs[i + 1]].copy() for i in range(len(sizes))]
        dg = [torch.from_numpy(a).cuda() for a in gl]
        zp.zero_grad_norm_overflow(dg, state, ws)
        zp.zero_adam_step(dg, dp, dm, dv, dl, ghp, state, ws)
        gst = zp.parse_state(state)
        st = oracle_step(gl, "f16", hp_, hm, hv, hl, "f16", ohp, sc, gst)
        assert_f32(torch.cat(dp).cpu().numpy(), np.concatenate(hp_), f"master step {k}", st.exact, bound_of(st, "p", 0))
        assert_f32(torch.cat(dm).cpu().numpy(), np.concatenate(hm), f"m step {k}", st.exact, bound_of(st, "m", 0))
        assert_f32(torch.cat(dv).cpu().numpy(), np.concatenate(hv), f"v step {k}", st.exact, bound_of(st, "v", 0))
        assert_lp(to_host(torch.cat(dl)), np.concatenate(hp_), "f16", f"p_lp step {k}", st.exact, bound_of(st, "p", 0))
