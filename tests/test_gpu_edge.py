"""GPU edge cases through the C ABI: every element-type pair on ragged sizes,
overflow at the first / last / tail position, loss-scale floor and growth,
empty shards, partition invariance over Nd emulated ranks, list versus flat,
run-to-run determinism, accumulation modes, and argument errors (each
rejected on the host before any launch)."""
import ctypes

import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import (bound_of, TORCH, assert_f32, assert_lp, assert_lp_copy, hp_pair, oracle_step, to_dev,  # noqa: E402
                        to_host)
from test_gpu_parity import run_full  # noqa: E402


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


PAIRS = [("f16", "f16"), ("bf16", "bf16"), ("f32", "bf16"), ("f32", "f16"), ("bf16", "f16"),
         ("f16", "bf16")]


@pytest.mark.parametrize("gdtype,pdtype", PAIRS)
@pytest.mark.parametrize("n", [1, 7, 8, 9, 17, 255, 2049, 65539, 1_000_003])
def test_ragged_sizes_all_types(zp, gdtype, pdtype, n):
    scale = 1.0 if gdtype != "f16" else 4096.0
    run_full(zp, n, gdtype, pdtype, 2, scale, max_norm=0.5 if n > 100 else 0.0, seed=n)


@pytest.mark.parametrize("where", ["first", "last", "tail", "middle"])
@pytest.mark.parametrize("nan", [False, True])
@pytest.mark.parametrize("gdtype", ["f16", "bf16", "f32"])
def test_overflow_positions(zp, where, nan, gdtype):
    n = 100_005  # 12,500 vectors of 8 and a tail of 5
    pos = {"first": 0, "last": n - 1, "tail": n - 3, "middle": 54_321}[where]
    scale = 65536.0 if gdtype == "f16" else 1.0
    st, skipped = run_full(zp, n, gdtype, "f16" if gdtype == "f16" else "bf16", 3, scale,
                           inf_step=1, inf_pos=pos, nan=nan)
    assert skipped == 1 and st["step"] == 2 and st["skipped"] == 1
    assert st["loss_scale"] == max(scale / 2, 1.0)


def test_overflow_on_first_step_then_recovery(zp):
    st, skipped = run_full(zp, 4099, "f16", "f16", 3, 1024.0, inf_step=0, inf_pos=4098)
    assert skipped == 1 and st["step"] == 2 and st["loss_scale"] == 512.0


def test_scale_floor_and_growth(zp):
    # floor: repeated overflow at scale 2 with floor 1
    st, _ = run_full(zp, 1000, "f16", "f16", 2, 2.0, inf_step=0, inf_pos=5)
    assert st["loss_scale"] == 1.0
    # growth after a window of 2 clean steps: 8 -> 16 -> 32
    st, _ = run_full(zp, 1000, "f16", "f16", 5, 8.0, hp_kw=dict(scale_window=2))
    assert st["loss_scale"] == 32.0 and st["good_steps"] == 1


def test_empty_shard(zp):
    state = zp.new_state(1024.0)
    ws = zp.new_workspace(1, 0)
    e16 = torch.empty(0, dtype=torch.float16, device="cuda")
    e32 = torch.empty(0, dtype=torch.float32, device="cuda")
    zp.zero_grad_norm_overflow(e16, state, ws)
    zp.zero_adam_step(e16, e32, e32, e32, e16, zp.HParams(), state, ws)
    st = zp.parse_state(state)
    assert st["step"] == 1 and st["last_norm"] == 0.0 and st["last_skipped"] == 0


def _shards(n_total, nd, align, seed):
    """Flat padded master/grad arrays of a layout and their per-rank views."""
    lay = oracle.partition_layout([n_total], nd, align)
    p0 = np.zeros(lay.padded_total, np.float32)
    p0[:n_total] = zs.host_master(n_total, seed)
    return lay, p0


@pytest.mark.parametrize("max_norm", [0.0, 0.3])
@pytest.mark.parametrize("mode", ["exchange", "accumulate"])
def test_partition_invariance(zp, max_norm, mode):
    """Nd = 4 emulated ranks on one GPU, each with its own shard, state and
    workspace.  The cross-rank sum of (sum g^2, found_inf) is done either by
    summing the ranks' 16-byte partials (what an all-reduce would do) or by
    the accumulate flag of pass 1.  With clipping off the concatenated shards
    equal the unpartitioned update bit for bit.  With clipping on the two
    norms are summed in different orders; each side is then checked against
    the oracle (bit for bit while its clip coefficient matches the oracle's,
    within the tolerance otherwise) and the norms must agree to 1e-8."""
    n_total, nd, align = 1_000_003, 4, 128
    lay, p0 = _shards(n_total, nd, align, 7)
    S = lay.shard_numel
    N = lay.padded_total
    ohp, ghp = hp_pair(max_norm=max_norm)
    scale = 1024.0
    full = dict(p=torch.from_numpy(p0.copy()).cuda(), m=torch.zeros(N, device="cuda"),
                v=torch.zeros(N, device="cuda"),
                lp=torch.zeros(N, dtype=torch.float16, device="cuda"),
                st=zp.new_state(scale), ws=zp.new_workspace(1, N))
    ranks = []
    for r in range(nd):
        ranks.append(dict(p=full["p"][r * S:(r + 1) * S].clone(),
                          m=torch.zeros(S, device="cuda"), v=torch.zeros(S, device="cuda"),
                          lp=torch.zeros(S, dtype=torch.float16, device="cuda"),
                          st=zp.new_state(scale), ws=zp.new_workspace(1, S)))
    # the oracle (unpartitioned: it runs on its own), once per side so that
    # each side's record of agreeing clip coefficients is its own
    ora = {side: dict(p=p0.copy(), m=np.zeros(N, np.float32), v=np.zeros(N, np.float32),
                      lp=np.zeros(N, np.uint16), sc=oracle.Scaler(loss_scale=scale))
           for side in ("full", "ranks")}
    last = {}
    for k in range(3):
        g = np.zeros(N, np.float16)
        g[:n_total] = zs.host_grad(n_total, 7, k, scale, "f16")
        dg = torch.from_numpy(g).cuda()
        zp.zero_grad_norm_overflow(dg, full["st"], full["ws"])
        zp.zero_adam_step(dg, full["p"], full["m"], full["v"], full["lp"], ghp, full["st"],
                          full["ws"])
        gs = [dg[r * S:(r + 1) * S] for r in range(nd)]
        if mode == "exchange":
            for r in range(nd):
                zp.zero_grad_norm_overflow(gs[r], ranks[r]["st"], ranks[r]["ws"])
            partial = sum(rk["st"][:16].view(torch.float64) for rk in ranks)
            for rk in ranks:
                rk["st"][:16] = partial.view(torch.uint8)
        else:
            for r in range(nd):
                zp.zero_grad_norm_overflow(gs[r], ranks[0]["st"], ranks[0]["ws"],
                                           accumulate=r > 0)
            for rk in ranks[1:]:
                rk["st"][:16] = ranks[0]["st"][:16]
        for r in range(nd):
            rk = ranks[r]
            zp.zero_adam_step(gs[r], rk["p"], rk["m"], rk["v"], rk["lp"], ghp, rk["st"], rk["ws"])
        fs = zp.parse_state(full["st"])
        rs = [zp.parse_state(rk["st"]) for rk in ranks]
        for x in rs:
            assert x["step"] == fs["step"] and x["loss_scale"] == fs["loss_scale"]
            assert x["last_clip"] == rs[0]["last_clip"] and x["last_norm"] == rs[0]["last_norm"]
            # binary32 partials grouped differently on each side: ~1e-9 apart
            assert abs(x["last_norm"] - fs["last_norm"]) <= 1e-8 * fs["last_norm"]
        for side, gst in (("full", fs), ("ranks", rs[0])):
            o = ora[side]
            last[side] = oracle_step([g], "f16", [o["p"]], [o["m"]], [o["v"]], [o["lp"]], "f16", ohp,
                                     o["sc"], gst)
    cat = {key: torch.cat([rk[key] for rk in ranks]) for key in ("p", "m", "v", "lp")}
    for key in ("p", "m", "v"):
        for side, got in (("full", full[key]), ("ranks", cat[key])):
            assert_f32(got.cpu().numpy(), ora[side][key], f"{side} {key}", last[side].exact,
                       bound_of(last[side], key, 0))
    for side, got in (("full", full["lp"]), ("ranks", cat["lp"])):
        assert_lp_copy(to_host(got), ora[side]["lp"], f"{side} p_lp", last[side].exact)
        assert_lp(to_host(got), ora[side]["p"], "f16", f"{side} p_lp", last[side].exact,
                  bound_of(last[side], "p", 0))
    if max_norm == 0.0:
        for key in ("p", "m", "v", "lp"):
            assert torch.equal(cat[key], full[key]), f"shards differ from the unpartitioned {key}"
    # the zero padding stays exactly zero
    assert not full["p"][n_total:].any() and not full["m"][n_total:].any()
    assert not full["v"][n_total:].any()


def test_list_equals_flat(zp):
    """One flat array versus the same elements cut into a list of arrays
    (ragged pieces): identical elementwise results, norms within 1e-8."""
    # 2047, 4094, 2041: a last 2048-element tile whose 8-element vectors and
    # scalar tail together need more threads than a block has
    sizes = [1, 9, 65536, 70001, 3, 131072 * 2 + 5, 8, 2047, 4094, 2041, 2048 * 3 + 2045]
    n = sum(sizes)
    ohp, ghp = hp_pair()
    p0 = zs.host_master(n, 3)
    flat = [torch.from_numpy(p0.copy()).cuda(), torch.zeros(n, device="cuda"),
            torch.zeros(n, device="cuda"), torch.zeros(n, dtype=torch.float16, device="cuda")]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    pieces = [[torch.from_numpy(p0[offs[i]:offs[i + 1]].copy()).cuda(),
               torch.zeros(sizes[i], device="cuda"), torch.zeros(sizes[i], device="cuda"),
               torch.zeros(sizes[i], dtype=torch.float16, device="cuda")] for i in range(len(sizes))]
    st_f, st_l = zp.new_state(256.0), zp.new_state(256.0)
    ws_f, ws_l = zp.new_workspace(1, n), zp.new_workspace(len(sizes), n)
    for k in range(3):
        g = zs.host_grad(n, 3, k, 256.0, "f16")
        dg = torch.from_numpy(g).cuda()
        gl = [torch.from_numpy(g[offs[i]:offs[i + 1]].copy()).cuda() for i in range(len(sizes))]
        zp.zero_grad_norm_overflow(dg, st_f, ws_f)
        zp.zero_adam_step(dg, *flat, ghp, st_f, ws_f)
        zp.zero_grad_norm_overflow(gl, st_l, ws_l)
        zp.zero_adam_step(gl, [q[0] for q in pieces], [q[1] for q in pieces],
                          [q[2] for q in pieces], [q[3] for q in pieces], ghp, st_l, ws_l)
        a, b = zp.parse_state(st_f), zp.parse_state(st_l)
        assert abs(a["last_norm"] - b["last_norm"]) <= 1e-8 * a["last_norm"]
    for j in range(4):
        cat = torch.cat([q[j] for q in pieces])
        assert torch.equal(cat, flat[j])


def test_run_to_run_determinism(zp):
    """Two runs of the same steps give the same bits, norm included."""
    n = 3_000_017
    outs = []
    for _ in range(2):
        _, ghp = hp_pair(max_norm=0.7)
        p = torch.from_numpy(zs.host_master(n, 11)).cuda()
        m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
        lp = torch.zeros(n, dtype=torch.float16, device="cuda")
        st, ws = zp.new_state(1024.0), zp.new_workspace(1, n)
        norms = []
        for k in range(3):
            dg = torch.from_numpy(zs.host_grad(n, 11, k, 1024.0, "f16")).cuda()
            zp.zero_grad_norm_overflow(dg, st, ws)
            zp.zero_adam_step(dg, p, m, v, lp, ghp, st, ws)
            norms.append(zp.parse_state(st)["last_norm"])
        outs.append((norms, p.cpu(), m.cpu(), v.cpu(), lp.cpu()))
    assert outs[0][0] == outs[1][0]
    for a, b in zip(outs[0][1:], outs[1][1:]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("gdtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("nb", [1, 2, 4, 8])
@pytest.mark.parametrize("overwrite", [True, False])
def test_accumulate(zp, gdtype, nb, overwrite):
    n = 200_003
    bufs = [zs.host_grad(n, 5, 0, 1.0, gdtype, micro=j) for j in range(nb)]
    acc0 = zs.host_normal(n, 1e-3, 5, "misc")
    ref = acc0.copy()
    oracle.accumulate(ref, bufs, gdtype, overwrite)
    dacc = torch.from_numpy(acc0.copy()).cuda()
    zp.zero_accumulate_grads(dacc, [to_dev(b, gdtype) for b in bufs], overwrite)
    assert dacc.cpu().numpy().tobytes() == ref.tobytes()


@pytest.mark.parametrize("gdtype,nb,overwrite,n", [
    ("f16", 1, True, 9), ("bf16", 4, True, 200_003), ("bf16", 4, False, 200_003), ("f32", 2, False, 65_541),
    ("f16", 8, True, 1_000_003), ("bf16", 4, True, 20_000_003)])
def test_accumulate_norm(zp, gdtype, nb, overwrite, n):
    """Accumulation fused with pass 1: the stored sums bit for bit as the
    oracle's accumulation, and the squared norm and overflow of the sums as
    the oracle's pass 1 over them, from a ragged 9 elements to 20,000,003
    (many iterations of the persistent grid)."""
    scale = 1024.0 if gdtype == "f16" else 1.0
    bufs = [zs.host_grad(n, 7, 0, scale, gdtype, micro=j) for j in range(nb)]
    acc0 = zs.host_normal(n, 1e-3, 7, "misc")
    ref = acc0.copy()
    oracle.accumulate(ref, bufs, gdtype, overwrite)
    sumsq, bad = oracle.norm_overflow([ref], "f32", scale)
    dacc = torch.from_numpy(acc0.copy()).cuda()
    st = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    zp.zero_accumulate_grads_norm(dacc, [to_dev(b, gdtype) for b in bufs], st, ws, overwrite)
    assert dacc.cpu().numpy().tobytes() == ref.tobytes()
    s = zp.parse_state(st)
    assert s["found_inf"] == float(bad) == 0.0
    assert abs(s["sumsq"] - sumsq) <= 1e-6 * sumsq
    # accumulate = True folds a second call (here overwriting acc) into the same sum
    ref2 = ref.copy()
    oracle.accumulate(ref2, bufs, gdtype, True)
    sumsq2, _ = oracle.norm_overflow([ref2], "f32", scale)
    zp.zero_accumulate_grads_norm(dacc, [to_dev(b, gdtype) for b in bufs], st, ws, True, accumulate=True)
    assert dacc.cpu().numpy().tobytes() == ref2.tobytes()
    assert abs(zp.parse_state(st)["sumsq"] - (sumsq + sumsq2)) <= 1e-6 * (sumsq + sumsq2)


@pytest.mark.parametrize("where", ["vector", "tail"])
def test_accumulate_norm_overflow(zp, where):
    n = 100_005
    bufs = [zs.host_grad(n, 8, 0, 1.0, "bf16", micro=j) for j in range(4)]
    pos = 4097 if where == "vector" else n - 2
    bufs[3].view(np.uint16)[pos] = 0x7F80  # +inf in the last micro-batch
    acc = torch.empty(n, device="cuda")
    st = zp.new_state(1.0)
    ws = zp.new_workspace(1, n)
    zp.zero_accumulate_grads_norm(acc, [to_dev(b, "bf16") for b in bufs], st, ws, True)
    assert zp.parse_state(st)["found_inf"] == 1.0
    assert np.isinf(acc.cpu().numpy()[pos])


def test_accumulate_norm_then_step_against_oracle(zp):
    """Three steps of four bf16 micro-batches with clipping: the fused
    accumulation + pass 1, then the decision and pass 2, every element of
    every step against the oracle's accumulation and step."""
    n, micro, seed = 300_007, 4, 31
    ohp, ghp = hp_pair(max_norm=0.05)
    p0 = zs.host_master(n, seed)
    dp = torch.from_numpy(p0.copy()).cuda()
    dm = torch.zeros(n, device="cuda")
    dv = torch.zeros(n, device="cuda")
    dlp = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
    dacc = torch.empty(n, device="cuda")
    state = zp.new_state(1.0)
    ws = zp.new_workspace(1, n)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    plp = np.zeros(n, np.uint16)
    sc = oracle.Scaler(loss_scale=1.0)
    for k in range(3):
        bufs = [zs.host_grad(n, seed, k, 1.0, "bf16", micro=j) for j in range(micro)]
        acc = np.zeros(n, np.float32)
        oracle.accumulate(acc, bufs, "bf16", True)
        zp.zero_accumulate_grads_norm(dacc, [to_dev(b, "bf16") for b in bufs], state, ws, True)
        zp.zero_adam_step(dacc, dp, dm, dv, dlp, ghp, state, ws)
        gst = zp.parse_state(state)
        st = oracle_step([acc], "f32", [p], [m], [v], [plp], "bf16", ohp, sc, gst)
        assert dacc.cpu().numpy().tobytes() == acc.tobytes()
        assert_f32(to_host(dp), p, f"master step {k}", st.exact, bound_of(st, "p", 0))
        assert_f32(to_host(dm), m, f"m step {k}", st.exact, bound_of(st, "m", 0))
        assert_f32(to_host(dv), v, f"v step {k}", st.exact, bound_of(st, "v", 0))
        assert_lp_copy(to_host(dlp), plp, f"p_lp step {k}", st.exact)
    assert zp.parse_state(state)["step"] == 3


def test_argument_errors_launch_nothing(zp):
    n = 4096
    g = torch.zeros(n + 8, dtype=torch.float16, device="cuda")
    p = torch.zeros(n + 8, device="cuda")
    m, v = torch.zeros(n, device="cuda"), torch.zeros(n, device="cuda")
    lp = torch.zeros(n, dtype=torch.float16, device="cuda")
    st = zp.new_state(1024.0)
    ws = zp.new_workspace(1, n)
    before = st.clone()
    hp = zp.HParams()
    with pytest.raises(zp.ZeroError) as e:  # grad starting 2 bytes off a 16-byte boundary
        zp.zero_grad_norm_overflow(g[1:n + 1], st, ws)
    assert e.value.code == -2
    with pytest.raises(zp.ZeroError) as e:
        zp.zero_adam_step(g[:n], p[1:n + 1], m, v, lp, hp, st, ws)
    assert e.value.code == -2
    with pytest.raises(zp.ZeroError) as e:  # sizes differ
        zp.zero_adam_step(g[:n], p[:n - 8], m, v, lp, hp, st, ws)
    assert e.value.code == -4
    with pytest.raises(zp.ZeroError) as e:  # master must be fp32
        zp.zero_adam_step(g[:n], g[:n], m, v, lp, hp, st, ws)
    assert e.value.code == -3
    with pytest.raises(zp.ZeroError) as e:  # low-precision copy must be 16-bit
        zp.zero_adam_step(g[:n], p[:n], m, v, p[:n], hp, st, ws)
    assert e.value.code == -3
    with pytest.raises(zp.ZeroError) as e:  # workspace too small
        zp.zero_grad_norm_overflow(g[:n], st, ws[:256])
    assert e.value.code == -5
    with pytest.raises(zp.ZeroError) as e:  # bad hyper-parameters
        zp.zero_adam_step(g[:n], p[:n], m, v, lp, zp.HParams(beta1=1.0), st, ws)
    assert e.value.code == -1
    with pytest.raises(zp.ZeroError) as e:  # a scale floor that is not a power of two
        zp.zero_step(g[:n], p[:n], m, v, lp, zp.HParams(min_scale=3.0), st, ws)
    assert e.value.code == -1
    # host memory passed through the raw C ABI is refused
    host = np.zeros(n, np.float16)
    lib = zp.lib()
    from zero_partitioned_mixed_layout_gb300.binding import _TList
    ptrs = (ctypes.c_void_p * 1)(host.ctypes.data)
    numel = (ctypes.c_int64 * 1)(n)
    tl = _TList(ptrs, numel, 1, 0)
    rc = lib.zero_grad_norm_overflow(ctypes.byref(tl), ctypes.c_void_p(st.data_ptr()), 0,
                                     ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -1
    torch.cuda.synchronize()
    assert torch.equal(st, before), "a rejected call changed the state"


@pytest.mark.parametrize("kind", ["flat", "list"])
@pytest.mark.parametrize("max_norm", [0.0, 0.3])
def test_fused_step_equals_split_calls(zp, kind, max_norm):
    """zero_step (pass 1, decision and pass 2 in one call, the kernels of a
    flat shard chained) gives the bits of zero_grad_norm_overflow followed by
    zero_adam_step, state included, over steps with and without overflow."""
    sizes = [1_000_003] if kind == "flat" else [5, 70_001, 3, 262_149, 8, 1, 4096, 2047, 6141]
    total = sum(sizes)
    p0 = zs.host_master(total, 21)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    _, ghp = hp_pair(max_norm=max_norm)

    def make():
        return dict(
            p=[torch.from_numpy(p0[offs[i]:offs[i + 1]].copy()).cuda() for i in range(len(sizes))],
            m=[torch.zeros(n, device="cuda") for n in sizes],
            v=[torch.zeros(n, device="cuda") for n in sizes],
            lp=[torch.zeros(n, dtype=torch.float16, device="cuda") for n in sizes],
            st=zp.new_state(1024.0), ws=zp.new_workspace(len(sizes), total))

    a, b = make(), make()
    for k in range(4):
        g = zs.host_grad(total, 21, k, zp.parse_state(a["st"])["loss_scale"], "f16")
        if k == 1:
            g[total - 2] = np.inf
        gl = [torch.from_numpy(g[offs[i]:offs[i + 1]].copy()).cuda() for i in range(len(sizes))]
        zp.zero_grad_norm_overflow(gl, a["st"], a["ws"])
        zp.zero_adam_step(gl, a["p"], a["m"], a["v"], a["lp"], ghp, a["st"], a["ws"])
        zp.zero_step(gl, b["p"], b["m"], b["v"], b["lp"], ghp, b["st"], b["ws"])
        torch.cuda.synchronize()
        assert torch.equal(a["st"], b["st"]), f"state differs at step {k}"
        for key in ("p", "m", "v", "lp"):
            for x, y in zip(a[key], b[key]):
                assert torch.equal(x, y), f"{key} differs at step {k}"
    st = zp.parse_state(b["st"])
    assert st["step"] == 3 and st["skipped"] == 1


@pytest.mark.parametrize("gdtype,pdtype", PAIRS)
@pytest.mark.parametrize("n", [1, 7, 8, 9, 2049, 65539, 1_000_003, (1 << 22) + 3])
def test_whole_step_call_against_oracle(zp, gdtype, pdtype, n):
    """zero_step on a flat shard (the three kernels chained) against the
    oracle, with clipping and an overflow step."""
    scale = 1.0 if gdtype != "f16" else 4096.0
    st, skipped = run_full(zp, n, gdtype, pdtype, 3, scale, max_norm=0.5 if n > 100 else 0.0, seed=n + 5,
                           inf_step=1, whole=True)
    assert skipped == 1 and st["step"] == 2


@pytest.mark.parametrize("where", ["first", "last", "tail"])
def test_whole_step_call_overflow_positions(zp, where):
    n = 100_005
    pos = {"first": 0, "last": n - 1, "tail": n - 3}[where]
    st, skipped = run_full(zp, n, "f16", "f16", 3, 65536.0, inf_step=2, inf_pos=pos, whole=True)
    assert skipped == 1 and st["step"] == 2 and st["loss_scale"] == 32768.0


def test_whole_step_call_many_steps_workspace_reuse(zp):
    """Twenty chained steps through one workspace: the reduction ticket and
    the bias-correction cache carry over from step to step."""
    n = 300_001
    st, skipped = run_full(zp, n, "bf16", "bf16", 20, 1.0, max_norm=0.2, seed=77, whole=True)
    assert skipped == 0 and st["step"] == 20


@pytest.mark.parametrize("kind", ["flat", "list"])
@pytest.mark.parametrize("gdtype", ["f16", "f32"])
def test_16_byte_aligned_state_matches_32(zp, kind, gdtype):
    """fp32 arrays that start on a 16- but not a 32-byte boundary take the
    16-byte access form of pass 2; it gives the bits of the 32-byte form."""
    sizes = [100_003] if kind == "flat" else [4099, 70_001, 2047]
    total = sum(sizes)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    p0 = zs.host_master(total, 51)
    _, ghp = hp_pair(max_norm=0.3)
    scale = 1024.0 if gdtype == "f16" else 1.0
    tdt = TORCH[gdtype]

    def make(shift):
        # `shift` floats into a 512-byte aligned allocation: 4 -> 16-byte aligned only
        def arr(n, fill=None, dtype=torch.float32):
            base = torch.zeros(n + 8, dtype=dtype, device="cuda")
            out = base[shift:shift + n]
            if fill is not None:
                out.copy_(fill)
            return out
        return dict(p=[arr(n, torch.from_numpy(p0[offs[i]:offs[i + 1]].copy())) for i, n in enumerate(sizes)],
                    m=[arr(n) for n in sizes], v=[arr(n) for n in sizes],
                    lp=[torch.zeros(n, dtype=torch.float16, device="cuda") for n in sizes],
                    st=zp.new_state(scale), ws=zp.new_workspace(len(sizes), total),
                    shift=shift, arr=arr)

    a32, a16 = make(0), make(4)
    assert a16["p"][0].data_ptr() % 32 == 16 and a32["p"][0].data_ptr() % 32 == 0
    for k in range(3):
        g = zs.host_grad(total, 51, k, scale, gdtype)
        gl = [torch.from_numpy(g[offs[i]:offs[i + 1]].copy()).cuda() for i in range(len(sizes))]
        for d in (a32, a16):
            gg = gl if gdtype != "f32" else [d["arr"](x.numel(), x, torch.float32) for x in gl]
            zp.zero_step(gg if kind == "list" else gg[0], d["p"] if kind == "list" else d["p"][0],
                         d["m"] if kind == "list" else d["m"][0], d["v"] if kind == "list" else d["v"][0],
                         d["lp"] if kind == "list" else d["lp"][0], ghp, d["st"], d["ws"])
        torch.cuda.synchronize()
        assert torch.equal(a32["st"], a16["st"])
        for key in ("p", "m", "v", "lp"):
            for x, y in zip(a32[key], a16[key]):
                assert torch.equal(x, y), f"{key} step {k}"


@pytest.mark.parametrize("whole", [True, False])
def test_learning_rate_schedule_and_beta_change(zp, whole):
    """Forty steps with the learning rate changed at every step (linear
    warm-up, then cosine decay), the betas changed at step 25 and an
    overflow at step 10.  The bias corrections come from the cached window
    of step counts (refilled every 16 steps and on the beta change), the
    step size from the cached 1 - beta1^t divided by the new rate on the
    device; every element of every step against the oracle (whole: through
    zero_step, else pass 1 and zero_adam_step)."""
    import math
    n, seed, scale = 50_001, 91, 1024.0
    p0 = zs.host_master(n, seed)
    dp = torch.from_numpy(p0.copy()).cuda()
    dm = torch.zeros(n, dtype=torch.float32, device="cuda")
    dv = torch.zeros(n, dtype=torch.float32, device="cuda")
    dlp = torch.zeros(n, dtype=torch.float16, device="cuda")
    state = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    plp = np.zeros(n, np.uint16)
    sc = oracle.Scaler(loss_scale=scale)
    skipped = 0
    for k in range(40):
        lr = 1e-3 * min(1.0, (k + 1) / 8) * 0.5 * (1.0 + math.cos(math.pi * k / 40))
        b1, b2 = (0.9, 0.999) if k < 25 else (0.85, 0.99)
        ohp, ghp = hp_pair(lr=lr, beta1=b1, beta2=b2, max_norm=0.5)
        g = zs.host_grad(n, seed, k, sc.loss_scale, "f16")
        if k == 10:
            g[zs.inf_index(n, seed, k)] = zs.host_cast(np.array([np.inf], np.float32), "f16")[0]
        dg = to_dev(g, "f16")
        if whole:
            zp.zero_step(dg, dp, dm, dv, dlp, ghp, state, ws)
        else:
            zp.zero_grad_norm_overflow(dg, state, ws)
            zp.zero_adam_step(dg, dp, dm, dv, dlp, ghp, state, ws)
        gst = zp.parse_state(state)
        st = oracle_step([g], "f16", [p], [m], [v], [plp], "f16", ohp, sc, gst)
        skipped += st.skip
        assert_f32(to_host(dp), p, f"master step {k}", st.exact, bound_of(st, "p", 0))
        assert_f32(to_host(dm), m, f"m step {k}", st.exact, bound_of(st, "m", 0))
        assert_f32(to_host(dv), v, f"v step {k}", st.exact, bound_of(st, "v", 0))
        assert_lp_copy(to_host(dlp), plp, f"p_lp step {k}", st.exact)
    assert skipped == 1 and zp.parse_state(state)["step"] == 39


def test_list_steps_from_two_host_threads(zp):
    """Two host threads issue list-mode steps at the same time, each on its
    own stream, workspace and tensors: their tables go through the shared
    pinned staging ring, and every result equals the same steps issued from
    one thread, bit for bit."""
    import threading

    sizes = [[4099, 70_001, 2047, 1], [333, 65_536, 12_345]]
    _, ghp = hp_pair(max_norm=0.3)

    def make(k):
        rng = np.random.default_rng(500 + k)
        return {
            "g": [[torch.from_numpy((rng.standard_normal(n) * 0.01).astype(np.float16)).cuda() for n in sizes[k]]
                  for _ in range(6)],
            "p": [torch.from_numpy(rng.standard_normal(n).astype(np.float32)).cuda() for n in sizes[k]],
            "m": [torch.zeros(n, device="cuda") for n in sizes[k]],
            "v": [torch.zeros(n, device="cuda") for n in sizes[k]],
            "lp": [torch.zeros(n, dtype=torch.float16, device="cuda") for n in sizes[k]],
            "st": zp.new_state(1.0), "ws": zp.new_workspace(len(sizes[k]), sum(sizes[k])),
        }

    def run(d, stream):
        with torch.cuda.stream(stream):
            for g in d["g"]:
                zp.zero_step(g, d["p"], d["m"], d["v"], d["lp"], ghp, d["st"], d["ws"], stream=stream)
        stream.synchronize()

    def result(d):
        return [to_host(t).tobytes() for t in d["p"] + d["m"] + d["v"] + d["lp"]] + [d["st"].cpu().numpy().tobytes()]

    alone = [make(0), make(1)]
    for d in alone:
        run(d, torch.cuda.Stream())
    both = [make(0), make(1)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    errors = []

    def worker(k):
        try:
            run(both[k], streams[k])
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k in range(2):
        assert result(both[k]) == result(alone[k]), f"thread {k}"
        assert zp.parse_state(both[k]["st"])["step"] == 6
