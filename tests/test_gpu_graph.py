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

from gpu_common import TORCH, assert_f32, assert_lp, hp_pair, oracle_step, to_dev, to_host  # noqa: E402


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
        assert_f32(to_host(dp), p, f"master step {k}")
        assert_f32(to_host(dm), m, f"m step {k}")
        assert_f32(to_host(dv), v, f"v step {k}")
        assert np.array_equal(to_host(dlp), plp), f"p_lp step {k}"
        assert_lp(to_host(dlp), p, pdtype, f"p_lp step {k}")
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
    previous one left."""
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
        ob, _ = oracle.onebit_server(hb, list(hs), f, scale=gs)
        assert to_host(d["es"]).tobytes() == f.tobytes(), f"server error, pass {r}"
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
