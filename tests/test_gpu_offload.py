"""The ZeRO-Offload step on a GB300 node: pass 1 on the GPU over the fp16
gradient, the gradient and state copied to the host, decision and update on
the host cores over host-resident fp32 state, the fp16 parameters and the
state copied back -- against the oracle, element by element."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import bound_of, assert_f32, assert_lp, assert_lp_copy, hp_pair, oracle_step, to_host  # noqa: E402


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


@pytest.mark.parametrize("max_norm", [0.0, 0.5])
def test_offload_step_against_oracle(zp, max_norm):
    n = 3_000_017
    scale = 4096.0
    ohp, ghp = hp_pair(max_norm=max_norm)
    d_state = zp.new_state(scale)
    ws = zp.new_workspace(1, n)
    h_state = torch.empty(zp.STATE_BYTES, dtype=torch.uint8, pin_memory=True)
    h_g = torch.empty(n, dtype=torch.float16, pin_memory=True)
    h_lp = torch.empty(n, dtype=torch.float16, pin_memory=True)
    d_lp = torch.zeros(n, dtype=torch.float16, device="cuda")
    p = torch.from_numpy(zs.host_master(n, 31))
    m, v = torch.zeros(n), torch.zeros(n)
    rp, rm, rv = p.numpy().copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    rlp = np.zeros(n, np.uint16)
    sc_o = oracle.Scaler(loss_scale=scale)
    for k in range(3):
        g = zs.host_grad(n, 31, k, sc_o.loss_scale, "f16")
        if k == 1:
            g[n - 1] = np.inf
        dg = torch.from_numpy(g).cuda()
        zp.zero_grad_norm_overflow(dg, d_state, ws)
        h_state.copy_(d_state)
        h_g.copy_(dg)
        sc = zp.zero_offload_decide(h_state, ghp)
        zp.zero_offload_apply(h_g, p, m, v, h_lp, sc)
        d_lp.copy_(h_lp)
        d_state.copy_(h_state)
        gst = zp.parse_state(h_state)
        ost = oracle_step([g], "f16", [rp], [rm], [rv], [rlp], "f16", ohp, sc_o, gst)
        assert_f32(p.numpy(), rp, f"master step {k}", ost.exact, bound_of(ost, "p", 0))
        assert_f32(m.numpy(), rm, f"m step {k}", ost.exact, bound_of(ost, "m", 0))
        assert_f32(v.numpy(), rv, f"v step {k}", ost.exact, bound_of(ost, "v", 0))
        assert_lp_copy(to_host(d_lp), rlp, f"fp16 params step {k}", ost.exact)
        assert_lp(to_host(d_lp), rp, "f16", f"fp16 params step {k}", ost.exact, bound_of(ost, "p", 0))
    st = zp.parse_state(d_state)
    assert st["step"] == 2 and st["skipped"] == 1 and st["loss_scale"] == scale / 2


@pytest.mark.parametrize("max_norm", [0.0, 0.5])
def test_state_in_pinned_host_memory(zp, max_norm):
    """master, m and v in pinned host memory (streamed by the GPU over the
    host link) give the bits of the same step with the state in HBM."""
    n = 2_000_003
    _, ghp = hp_pair(max_norm=max_norm)
    p0 = zs.host_master(n, 33)
    dev = dict(p=torch.from_numpy(p0.copy()).cuda(), m=torch.zeros(n, device="cuda"),
               v=torch.zeros(n, device="cuda"), lp=torch.zeros(n, dtype=torch.float16, device="cuda"),
               st=zp.new_state(1024.0), ws=zp.new_workspace(1, n))
    host = dict(p=torch.from_numpy(p0.copy()).pin_memory(), m=torch.zeros(n).pin_memory(),
                v=torch.zeros(n).pin_memory(), lp=torch.zeros(n, dtype=torch.float16, device="cuda"),
                st=zp.new_state(1024.0), ws=zp.new_workspace(1, n))
    for k in range(3):
        g = zs.host_grad(n, 33, k, zp.parse_state(dev["st"])["loss_scale"], "f16")
        if k == 1:
            g[5] = np.nan
        dg = torch.from_numpy(g).cuda()
        for d in (dev, host):
            zp.zero_step(dg, d["p"], d["m"], d["v"], d["lp"], ghp, d["st"], d["ws"])
        torch.cuda.synchronize()
        assert torch.equal(dev["st"], host["st"])
        for key in ("p", "m", "v"):
            assert torch.equal(dev[key].cpu(), host[key]), f"{key} step {k}"
        assert torch.equal(dev["lp"], host["lp"])
    # pageable host memory is refused
    with pytest.raises(zp.ZeroError):
        from zero_partitioned_mixed_layout_gb300.binding import _TList, _HParams  # noqa: F401
        pageable = torch.zeros(n)
        lib = zp.lib()
        import ctypes
        def tl(t, code):
            ptrs = (ctypes.c_void_p * 1)(t.data_ptr())
            numel = (ctypes.c_int64 * 1)(t.numel())
            return _TList(ptrs, numel, 1, code), ptrs, numel
        a = [tl(x, c) for x, c in ((dg, 0), (pageable, 2), (host["m"], 2), (host["v"], 2), (host["lp"], 0))]
        h = ghp._c()
        rc = lib.zero_adam_step(*[ctypes.byref(x[0]) for x in a], ctypes.byref(h),
                                ctypes.c_void_p(host["st"].data_ptr()), ctypes.c_void_p(host["ws"].data_ptr()),
                                host["ws"].numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        zp.binding._check(rc, "zero_adam_step")
