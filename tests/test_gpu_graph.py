"""CUDA graphs: a step captured once and replayed, against the oracle step
by step (the device state -- loss scale, step count, norm, the cache of the
next step's bias corrections -- moves on at every replay as over calls issued
one by one), and the calls that copy a host-built table refused under
capture (ZERO_ECAPTURE) with nothing enqueued."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import bound_of, TORCH, assert_f32, assert_lp, assert_lp_copy, hp_pair, oracle_step, to_dev, to_host  # noqa: E402


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("gdtype,pdtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", "f16")])
def test_flat_step_graph_replays_match_oracle(zp, gdtype, pdtype):
    """zero_step on a flat shard: one eager step, then the call captured and
    replayed five times with a new gradient copied into the captured buffer
    before each replay (an overflow in replay 3); every element of every
    step against the oracle."""
    n, seed = 300_001, 17
    scale = 1.0 if gdtype != "f16" else 4096.0
    ohp, ghp = hp_pair(max_norm=0.5)
    p0 = zs.host_master(n, seed)
    dp = torch.from_numpy(p0.copy()).cuda()
    dm = torch.zeros(n, dtype=torch.float32, device="cuda")
    dv = torch.zeros(n, dtype=torch.float32, device="cuda")
    dlp = torch.zeros(n, dtype=TORCH[pdtype], device="cuda")
    dg = torch.zeros(n, dtype=TORCH[gdtype], device="cuda")
    state = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    plp = np.zeros(n, np.uint16)
    sc = oracle.Scaler(loss_scale=scale)

    def step():
        zp.zero_step(dg, dp, dm, dv, dlp, ghp, state, ws)

    graph = None
    skipped = 0
    for k in range(6):
        g = zs.host_grad(n, seed, k, sc.loss_scale, gdtype)
        if k == 3:
            g[zs.inf_index(n, seed, k)] = zs.host_cast(np.array([np.inf], np.float32), gdtype)[0]
        dg.copy_(to_dev(g, gdtype))
        if k == 0:
            step()  # eager: also loads the kernels before the capture
        else:
            if graph is None:
                graph = capture(step)
                # capturing ran nothing
                assert zp.parse_state(state)["step"] == 1
            graph.replay()
        torch.cuda.synchronize()
        gst = zp.parse_state(state)
        st = oracle_step([g], gdtype, [p], [m], [v], [plp], pdtype, ohp, sc, gst)
        skipped += st.skip
        assert_f32(to_host(dp), p, f"master step {k}", st.exact, bound_of(st, "p", 0))
        assert_f32(to_host(dm), m, f"m step {k}", st.exact, bound_of(st, "m", 0))
        assert_f32(to_host(dv), v, f"v step {k}", st.exact, bound_of(st, "v", 0))
        assert_lp_copy(to_host(dlp), plp, f"p_lp step {k}", st.exact)
        assert_lp(to_host(dlp), p, pdtype, f"p_lp step {k}", st.exact, bound_of(st, "p", 0))
    st = zp.parse_state(state)
    assert skipped == 1 and st["step"] == 5 and st["skipped"] == 1


def test_list_step_refused_under_capture(zp):
    """A list of several arrays copies its table into the workspace: under
    capture the call returns ZERO_ECAPTURE and enqueues nothing (the graph
    holds only the other work captured with it); outside capture it runs."""
    sizes = [1000, 2048, 77]
    ohp, ghp = hp_pair()
    gs = [torch.ones(k, dtype=torch.float16, device="cuda") for k in sizes]
    ps = [torch.ones(k, dtype=torch.float32, device="cuda") for k in sizes]
    ms = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in sizes]
    vs = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in sizes]
    state = zp.new_state(1.0)
    ws = zp.new_workspace(len(sizes), sum(sizes))
    marker = torch.zeros(1, device="cuda")
    errors = []

    def body():
        marker.add_(1.0)
        try:
            zp.zero_step(gs, ps, ms, vs, None, ghp, state, ws)
        except zp.ZeroError as e:
            errors.append(e)

    # kernels loaded before the capture
    zp.zero_grad_norm_overflow(gs[0], state, ws)
    torch.cuda.synchronize()
    before = [to_host(t).tobytes() for t in ps]
    graph = capture(body)
    assert len(errors) == 1 and errors[0].code == zp.ZERO_ECAPTURE
    graph.replay()
    torch.cuda.synchronize()
    assert float(marker[0]) == 1.0
    assert [to_host(t).tobytes() for t in ps] == before
    assert zp.parse_state(state)["step"] == 0
    zp.zero_step(gs, ps, ms, vs, None, ghp, state, ws)
    torch.cuda.synchronize()
    assert zp.parse_state(state)["step"] == 1


def _server_inputs(zp, nd, S, seed, T=10):
    rng = np.random.default_rng(seed)
    w = S // 32
    hb = [rng.integers(0, 2 ** 32, w, dtype=np.uint64).astype(np.uint32) for _ in range(nd)]
    hs = rng.uniform(1e-4, 1.1e-3, nd).astype(np.float32)
    hf = (rng.standard_normal(S) * 1e-4).astype(np.float32)
    st = zp.binding._State()
    zp.binding.lib().zero_state_init(zp.binding.ctypes.byref(st), 1024.0)
    st.step = T
    raw = bytes(zp.binding.ctypes.string_at(zp.binding.ctypes.byref(st), zp.STATE_BYTES))
    d = {
        "wbits": [torch.from_numpy(b.view(np.int32)).cuda() for b in hb],
        "wscale": torch.from_numpy(hs).cuda(),
        "es": torch.from_numpy(hf.copy()).cuda(),
        "bits": torch.zeros(w, dtype=torch.int32, device="cuda"),
        "scale": torch.zeros(1, dtype=torch.float32, device="cuda"),
        "state": torch.frombuffer(bytearray(raw), dtype=torch.uint8).cuda(),
        "ws": zp.new_workspace(nd, nd * S),
    }
    z = torch.zeros(32, dtype=torch.float32, device="cuda")
    zp.zero_onebit_worker(torch.zeros(32, dtype=torch.float16, device="cuda"), z, z.clone(),
                          torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.zeros(1, dtype=torch.float32, device="cuda"), zp.HParams(), T,
                          d["state"], d["ws"])
    return hb, hs, hf, d


def test_onebit_server_graph_replay(zp):
    """The 1-bit server pass (pointers as a launch argument) captured and
    replayed twice: each replay is the oracle's server pass on the error the
    previous one left (which the GPU holds in deferred form)."""
    nd, S = 16, 65_536
    hb, hs, hf, d = _server_inputs(zp, nd, S, 5)

    def server():
        zp.zero_onebit_server(d["wbits"], d["wscale"], d["es"], d["bits"], d["scale"], d["ws"])

    server()
    torch.cuda.synchronize()
    graph = capture(server)
    f = hf.copy()
    for r in range(3):
        if r:
            graph.replay()
            torch.cuda.synchronize()
        gs = float(d["scale"][0])
        x = np.empty(S, np.float32)
        ob, _ = oracle.onebit_server(hb, list(hs), f, scale=gs, x_out=x)
        # the GPU keeps the compressed value (its error in deferred form)
        assert to_host(d["es"]).tobytes() == x.tobytes(), f"server input, pass {r}"
        assert np.array_equal(d["bits"].cpu().numpy().view(np.uint32), ob), f"server signs, pass {r}"


def test_onebit_server_table_refused_under_capture(zp):
    """More than 256 workers: the pointers go as a workspace table, which a
    capture refuses."""
    nd, S = 257, 1024
    _, _, hf, d = _server_inputs(zp, nd, S, 6)
    errors = []

    def server():
        try:
            zp.zero_onebit_server(d["wbits"], d["wscale"], d["es"], d["bits"], d["scale"], d["ws"])
        except zp.ZeroError as e:
            errors.append(e)

    marker = torch.zeros(1, device="cuda")

    def body():
        marker.add_(1.0)
        server()

    graph = capture(body)
    assert len(errors) == 1 and errors[0].code == zp.ZERO_ECAPTURE
    graph.replay()
    torch.cuda.synchronize()
    assert to_host(d["es"]).tobytes() == hf.tobytes()


def test_gather_graph_replay(zp):
    """The stage-3 gather (at most 64 tensors: the entries travel as a launch
    argument) captured and replayed after the shards change."""
    numel = [1000, 37, 4096, 5, 12_345]
    nd, align = 4, 128
    lay = zp.zero_partition_layout(numel, nd, align)
    S = lay.shard_numel
    flat = torch.arange(nd * S, dtype=torch.float32, device="cuda").to(torch.float16)
    shards = [flat[r * S:(r + 1) * S].clone() for r in range(nd)]
    outs = [torch.zeros(k, dtype=torch.float16, device="cuda") for k in numel]
    ws = torch.zeros(zp.zero_gather_workspace_bytes(len(numel), nd), dtype=torch.uint8, device="cuda")

    def gather():
        zp.zero_gather_params(shards, outs, lay.tensor_offset, ws)

    gather()
    torch.cuda.synchronize()
    graph = capture(gather)
    for s in shards:
        s.mul_(-1.0)
    graph.replay()
    torch.cuda.synchronize()
    full = torch.cat(shards)
    for t, off, k in zip(outs, lay.tensor_offset, numel):
        assert torch.equal(t, full[off:off + k])


def _list_case(sizes, gdtype, pdtype, seed, scale):
    rng = np.random.default_rng(seed)
    d = {
        "p": [torch.from_numpy(rng.standard_normal(n).astype(np.float32) * 0.02).cuda() for n in sizes],
        "m": [torch.zeros(n, device="cuda") for n in sizes],
        "v": [torch.zeros(n, device="cuda") for n in sizes],
        "lp": [torch.zeros(n, dtype=TORCH[pdtype], device="cuda") for n in sizes],
        "g": [torch.zeros(n, dtype=TORCH[gdtype], device="cuda") for n in sizes],
    }
    return d


def _grads(sizes, gdtype, seed, k, scale, inf=False):
    out = [zs.host_grad(n, seed + i, k, scale, gdtype) for i, n in enumerate(sizes)]
    if inf:
        out[1][7] = zs.host_cast(np.array([np.inf], np.float32), gdtype)[0]
    return out


@pytest.mark.parametrize("gdtype,pdtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", "f16")])
def test_prepared_list_step_equals_zero_step(zp, gdtype, pdtype):
    """A prepared list step gives zero_step's results bit for bit, step
    after step (an overflow in step 2), with the table copied once."""
    sizes = [4099, 70_001, 2047, 1, 12_345]
    scale = 1024.0 if gdtype == "f16" else 1.0
    _, ghp = hp_pair(max_norm=0.3)
    a, b = _list_case(sizes, gdtype, pdtype, 1, scale), _list_case(sizes, gdtype, pdtype, 1, scale)
    sa, sb = zp.new_state(scale), zp.new_state(scale)
    wa, wb = zp.new_workspace(len(sizes), sum(sizes)), zp.new_workspace(len(sizes), sum(sizes))
    plan = zp.zero_list_prepare(b["g"], b["p"], b["m"], b["v"], b["lp"], wb)
    assert plan.n == len(sizes)
    for k in range(4):
        hg = _grads(sizes, gdtype, 40, k, scale, inf=(k == 2))
        for t, x in zip(a["g"], hg):
            t.copy_(to_dev(x, gdtype))
        for t, x in zip(b["g"], hg):
            t.copy_(to_dev(x, gdtype))
        zp.zero_step(a["g"], a["p"], a["m"], a["v"], a["lp"], ghp, sa, wa)
        zp.zero_step_prepared(plan, ghp, sb, wb)
        torch.cuda.synchronize()
        for key in ("p", "m", "v", "lp"):
            for x, y in zip(a[key], b[key]):
                assert to_host(x).tobytes() == to_host(y).tobytes(), f"{key} step {k}"
        assert sa.cpu().numpy().tobytes() == sb.cpu().numpy().tobytes()
    assert zp.parse_state(sb)["step"] == 3 and zp.parse_state(sb)["skipped"] == 1


def test_prepared_list_step_graph_replays_match_oracle(zp):
    """A list step prepared once, then captured and replayed four times with
    new gradients copied into the captured tensors: every element of every
    step against the oracle."""
    sizes = [4099, 70_001, 2047, 1, 12_345]
    gdtype, pdtype, scale = "f16", "f16", 4096.0
    ohp, ghp = hp_pair(max_norm=0.3)
    d = _list_case(sizes, gdtype, pdtype, 2, scale)
    host = {"p": [to_host(t).copy() for t in d["p"]], "m": [np.zeros(n, np.float32) for n in sizes],
            "v": [np.zeros(n, np.float32) for n in sizes], "lp": [np.zeros(n, np.uint16) for n in sizes]}
    state = zp.new_state(scale)
    ws = zp.new_workspace(len(sizes), sum(sizes))
    plan = zp.zero_list_prepare(d["g"], d["p"], d["m"], d["v"], d["lp"], ws)
    zp.zero_grad_norm_overflow(d["g"][0], zp.new_state(scale), zp.new_workspace(1, sizes[0]))  # kernels loaded
    torch.cuda.synchronize()
    graph = capture(lambda: zp.zero_step_prepared(plan, ghp, state, ws))
    assert zp.parse_state(state)["step"] == 0
    sc = oracle.Scaler(loss_scale=scale)
    for k in range(4):
        hg = _grads(sizes, gdtype, 50, k, sc.loss_scale, inf=(k == 1))
        for t, x in zip(d["g"], hg):
            t.copy_(to_dev(x, gdtype))
        graph.replay()
        torch.cuda.synchronize()
        gst = zp.parse_state(state)
        st = oracle_step(hg, gdtype, host["p"], host["m"], host["v"], host["lp"], pdtype, ohp, sc, gst)
        for i in range(len(sizes)):
            assert_f32(to_host(d["p"][i]), host["p"][i], f"master {i} step {k}", st.exact, bound_of(st, "p", i))
            assert_f32(to_host(d["m"][i]), host["m"][i], f"m {i} step {k}", st.exact, bound_of(st, "m", i))
            assert_f32(to_host(d["v"][i]), host["v"][i], f"v {i} step {k}", st.exact, bound_of(st, "v", i))
            assert_lp_copy(to_host(d["lp"][i]), host["lp"][i], f"p_lp {i} step {k}", st.exact)
    assert zp.parse_state(state)["step"] == 3


def test_prepare_refused_under_capture_and_plan_checks(zp):
    """Preparing copies a table: refused under capture.  A plan runs only in
    the workspace it was prepared in.  A one-array plan runs zero_step."""
    sizes = [1000, 2048]
    _, ghp = hp_pair()
    d = _list_case(sizes, "f16", "f16", 3, 1.0)
    ws = zp.new_workspace(len(sizes), sum(sizes))
    errors = []

    def body():
        try:
            zp.zero_list_prepare(d["g"], d["p"], d["m"], d["v"], d["lp"], ws)
        except zp.ZeroError as e:
            errors.append(e)
        marker.add_(1.0)

    marker = torch.zeros(1, device="cuda")
    capture(body)
    assert len(errors) == 1 and errors[0].code == zp.ZERO_ECAPTURE
    plan = zp.zero_list_prepare(d["g"], d["p"], d["m"], d["v"], d["lp"], ws)
    other = zp.new_workspace(len(sizes), sum(sizes))
    with pytest.raises(zp.ZeroError) as e:
        zp.zero_step_prepared(plan, ghp, zp.new_state(1.0), other)
    assert e.value.code == -1
    # one array
    n = 50_001
    one = _list_case([n], "bf16", "bf16", 4, 1.0)
    two = _list_case([n], "bf16", "bf16", 4, 1.0)
    hg = _grads([n], "bf16", 60, 0, 1.0)
    one["g"][0].copy_(to_dev(hg[0], "bf16"))
    two["g"][0].copy_(to_dev(hg[0], "bf16"))
    s1, s2 = zp.new_state(1.0), zp.new_state(1.0)
    w1, w2 = zp.new_workspace(1, n), zp.new_workspace(1, n)
    p1 = zp.zero_list_prepare(one["g"], one["p"], one["m"], one["v"], one["lp"], w1)
    zp.zero_step_prepared(p1, ghp, s1, w1)
    zp.zero_step(two["g"][0], two["p"][0], two["m"][0], two["v"][0], two["lp"][0], ghp, s2, w2)
    torch.cuda.synchronize()
    for key in ("p", "m", "v", "lp"):
        assert to_host(one[key][0]).tobytes() == to_host(two[key][0]).tobytes(), key
