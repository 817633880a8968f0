"""1-bit Adam's compression stage on one GPU against the oracle: the Nd
workers, the Nd servers and the update of one compression-stage step, each
worker and server as the rank it would be (its own state and workspace).
Two comparisons: the oracle running on its own for several steps, every
value within bounds derived from the two sides' norm summation orders
(test_onebit_free_running_against_oracle); and, for the element arithmetic
itself, the oracle handed the GPU's scales, bit for bit (the binary64 norm
is summed in another order: the scales agree within 2^-22).  Also the
benchmark's full-size step on sampled elements plus the norm property.

The GPU holds each error in deferred form (the compression's input x and
its scale s; the error is x - s*sign(x)); the oracle holds it explicitly.
The tests compare the GPU's x with the oracle's compressed value and the
error the pair (x, s) stands for with the oracle's error, bit for bit."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import TORCH, to_dev, to_host  # noqa: E402

SCALE_REL = 2.0 ** -22


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def state_at(zp, loss_scale, step):
    """A device state after `step` applied warm-up steps."""
    st = zp.binding._State()
    zp.binding.lib().zero_state_init(zp.binding.ctypes.byref(st), float(loss_scale))
    st.step = int(step)
    raw = bytes(zp.binding.ctypes.string_at(zp.binding.ctypes.byref(st), zp.STATE_BYTES))
    return torch.frombuffer(bytearray(raw), dtype=torch.uint8).cuda()


def words(t):
    return t.cpu().numpy().view(np.uint32)


def bit_at(w, idx):
    """Sign bits of elements idx from packed words (bit k of word j is
    element 32j + k)."""
    return ((w[idx >> 5] >> (idx & 31).astype(np.uint32)) & 1).astype(np.uint8)


def deferred_error(x, s):
    """The error a compression with input x (float32) and scale s left:
    x - s where x is not negative (-0 included), x + s elsewhere; one
    binary32 rounding."""
    s = np.float32(s)
    return np.where(x < 0, x + s, x - s).astype(np.float32)


def pack(b):
    """Bits (one per element, in order) to packed words."""
    b = np.pad(np.asarray(b, np.uint8), (0, (-len(b)) % 32))
    return np.packbits(b, bitorder="little").view(np.uint32)


def run_gpu_step(zp, d, nd, S, numel, hp, T, pdtype, compressed=False):
    """One compression-stage step of every rank on the device arrays in d.
    compressed: the workers read the momentum as the previous step's server
    signs and scales, and the update leaves the dense m alone."""
    n = nd * S
    for i in range(nd):
        for k in range(nd):
            zp.zero_grad_norm_overflow(d["g"][k], d["state"][i], d["ws"][i], accumulate=k > 0)
    mom = (d["sbits"].clone(), d["sscale"].clone()) if compressed else d["m"]
    for i in range(nd):
        zp.zero_onebit_worker(d["g"][i], mom, d["ew"][i], d["wbits"][i], d["wscale"][i:i + 1], hp, T,
                              d["state"][i], d["ws"][i])
    w = S // 32
    for j in range(nd):
        zp.zero_onebit_server([d["wbits"][i][j * w:(j + 1) * w] for i in range(nd)], d["wscale"], d["es"][j],
                              d["sbits"][j * w:(j + 1) * w], d["sscale"][j:j + 1], d["ws"][j])
    zp.zero_onebit_update(d["sbits"], d["sscale"], S, numel, d["p"], None if compressed else d["m"], d["v"],
                          d["plp"], d["ws"][0])
    torch.cuda.synchronize()
    assert n == d["p"].numel()


def setup(zp, nd, S, gdtype, pdtype, seed, loss_scale, T, inf_at=None):
    n = nd * S
    rng = np.random.default_rng(seed)
    h = {
        "g": [zs.host_grad(n, seed + i, 0, loss_scale, gdtype) for i in range(nd)],
        "p": zs.host_master(n, seed),
        "m": (rng.standard_normal(n) * 1e-3).astype(np.float32),
        "v": (rng.uniform(0.1, 1.0, n) * 1e-6).astype(np.float32),
        # the errors in the GPU's deferred form: inputs and scales of a
        # previous compression
        "xw": [(rng.standard_normal(n) * 1e-4).astype(np.float32) for _ in range(nd)],
        "xs": [(rng.standard_normal(S) * 1e-4).astype(np.float32) for _ in range(nd)],
        "sw": rng.uniform(1e-5, 1e-4, nd).astype(np.float32),
        "ss": rng.uniform(1e-5, 1e-4, nd).astype(np.float32),
    }
    # the same errors, explicit, for the oracle
    h["ew"] = [deferred_error(x, s) for x, s in zip(h["xw"], h["sw"])]
    h["es"] = [deferred_error(x, s) for x, s in zip(h["xs"], h["ss"])]
    if inf_at is not None:
        g = h["g"][inf_at[0]]
        (g.view(np.uint16) if gdtype != "f32" else g.view(np.uint32))[inf_at[1]] = \
            {"f16": 0x7C00, "bf16": 0x7F80, "f32": 0x7F800000}[gdtype]
    h["plp"] = oracle.to_lp(h["p"], pdtype) if pdtype else None
    d = {
        "g": [to_dev(g, gdtype) for g in h["g"]],
        "p": to_dev(h["p"], "f32"), "m": to_dev(h["m"], "f32"), "v": to_dev(h["v"], "f32"),
        "ew": [to_dev(x, "f32") for x in h["xw"]], "es": [to_dev(x, "f32") for x in h["xs"]],
        "plp": (to_dev(h["plp"].view(np.float16) if pdtype == "f16" else h["plp"], pdtype)
                if pdtype else None),
        "wbits": [torch.zeros(n // 32, dtype=torch.int32, device="cuda") for _ in range(nd)],
        "wscale": torch.from_numpy(h["sw"].copy()).cuda(),
        "sbits": torch.zeros(n // 32, dtype=torch.int32, device="cuda"),
        "sscale": torch.from_numpy(h["ss"].copy()).cuda(),
        "state": [state_at(zp, loss_scale, T) for _ in range(nd)],
        "ws": [zp.new_workspace(1, n) for _ in range(nd)],
    }
    return h, d


def check_step(zp, h, d, nd, S, numel, gdtype, pdtype, hp, sc, T, dense_m=True):
    """Runs the oracle's step with the GPU's scales and compares everything
    (the dense m only when the GPU wrote it)."""
    ew0 = [e.copy() for e in h["ew"]]
    # the scales the oracle computes itself agree with the GPU's closely
    free = oracle.onebit_step(h["g"], gdtype, S, numel, h["p"].copy(), h["m"].copy(), h["v"],
                              [e.copy() for e in h["ew"]], [e.copy() for e in h["es"]], None, "f16", hp,
                              oracle.Scaler(sc.loss_scale, sc.step, sc.good_steps), T)
    gw = d["wscale"].cpu().numpy()
    gs = d["sscale"].cpu().numpy()
    st0 = zp.parse_state(d["state"][0])
    res = oracle.onebit_step(h["g"], gdtype, S, numel, h["p"], h["m"], h["v"], h["ew"], h["es"], h["plp"],
                             pdtype or "f16", hp, sc, T, worker_scales=list(gw), server_scales=list(gs),
                             clip=st0["last_clip"])
    for i in range(nd):
        st = zp.parse_state(d["state"][i])
        assert bool(st["last_skipped"]) == res.step.skip and st["step"] == sc.step
        assert st["loss_scale"] == sc.loss_scale
    if res.step.skip:
        return res
    for i in range(nd):
        assert abs(gw[i] - free.worker_scales[i]) <= SCALE_REL * free.worker_scales[i], f"worker {i} scale"
        assert np.array_equal(words(d["wbits"][i]), res.worker_bits[i]), f"worker {i} signs"
        x = to_host(d["ew"][i])
        assert x.tobytes() == res.worker_x[i].tobytes(), f"worker {i} compressed value"
        assert deferred_error(x, gw[i]).tobytes() == h["ew"][i].tobytes(), f"worker {i} error"
    for j in range(nd):
        assert abs(gs[j] - free.server_scales[j]) <= 4 * SCALE_REL * free.server_scales[j], f"server {j} scale"
        x = to_host(d["es"][j])
        assert x.tobytes() == res.server_x[j].tobytes(), f"server {j} compressed value"
        assert deferred_error(x, gs[j]).tobytes() == h["es"][j].tobytes(), f"server {j} error"
    assert np.array_equal(words(d["sbits"]), np.concatenate(res.server_bits))
    assert to_host(d["p"]).tobytes() == h["p"].tobytes(), "master"
    if dense_m:
        assert to_host(d["m"]).tobytes() == h["m"].tobytes(), "momentum"
    if pdtype:
        assert np.array_equal(to_host(d["plp"]), h["plp"]), "low-precision params"
    assert any((e != e0).any() for e, e0 in zip(h["ew"], ew0))
    return res


@pytest.mark.parametrize("nd,S", [(1, 1024), (2, 2048), (3, 4096), (4, 65_536), (16, 8192)])
@pytest.mark.parametrize("gdtype,pdtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", None)])
def test_onebit_step_matches_oracle(zp, nd, S, gdtype, pdtype):
    T = 100
    scale = 1.0 if gdtype == "bf16" else 1024.0
    h, d = setup(zp, nd, S, gdtype, pdtype, 7 * nd + S, scale, T)
    numel = nd * S - 13
    hp = oracle.HParams()
    zhp = zp.HParams()
    run_gpu_step(zp, d, nd, S, numel, zhp, T, pdtype)
    check_step(zp, h, d, nd, S, numel, gdtype, pdtype, hp, oracle.Scaler(scale, T), T)


def test_onebit_three_steps_with_clipping(zp):
    nd, S, T = 4, 4096, 20
    h, d = setup(zp, nd, S, "f16", "f16", 99, 1024.0, T)
    hp = oracle.HParams(max_norm=0.05)
    zhp = zp.HParams(max_norm=0.05)
    sc = oracle.Scaler(1024.0, T)
    for step in range(3):
        for i in range(nd):
            h["g"][i] = zs.host_grad(nd * S, 500 + 10 * step + i, step, 1024.0, "f16")
            d["g"][i] = to_dev(h["g"][i], "f16")
        run_gpu_step(zp, d, nd, S, nd * S, zhp, T, "f16")
        res = check_step(zp, h, d, nd, S, nd * S, "f16", "f16", hp, sc, T)
        assert res.step.scalars["clip"] < 1.0


U = 2.0 ** -24        # binary32 unit roundoff
TINY = 2.0 ** -147    # a few subnormal ulps: the floor of any rounding allowance


def _abs(a):
    return np.abs(np.asarray(a, np.float64))


@pytest.mark.parametrize("nd,S", [(4, 4096), (16, 2048)])
@pytest.mark.parametrize("gdtype,pdtype,max_norm", [("f16", "f16", 0.0), ("bf16", "bf16", 0.05)])
def test_onebit_free_running_against_oracle(zp, nd, S, gdtype, pdtype, max_norm):
    """Three compression-stage steps on the GPU and in the oracle, each side
    taking its own decision, norms and scales: nothing the GPU computes goes
    into the oracle.  The two sides sum the norms in different orders, so
    their binary32 scales may differ in the last places; through the error
    feedback that difference reaches the next step's inputs, and where a
    compressed value lies within it of zero its sign may come out the other
    way.  Each step is held to the bounds this implies, derived from the
    differences that enter the step (rounding allowances of a few ulps per
    operation where an input differs):
      * every compressed value x (worker) and y (server) within the bound
        carried through its arithmetic from the entering differences;
      * every scale within the difference of the inputs' L2 norms (the
        triangle inequality) plus the summation-order allowance;
      * a sign different from the oracle's only where |x| (|y|) is within
        its bound;
      * every error, momentum and master within what these imply.
    (A server's scale is shared by its whole chunk, so a last-place
    difference in it moves every element's momentum and master a little:
    the bounds above, not a flat relative bar, are the measure.)  Sign
    flips must stay rare."""
    T, steps = 50, 3
    scale = 1.0 if gdtype == "bf16" else 1024.0
    h, d = setup(zp, nd, S, gdtype, pdtype, 900 + nd, scale, T)
    n, numel = nd * S, nd * S - 11
    hp, zhp = oracle.HParams(max_norm=max_norm), zp.HParams(max_norm=max_norm)
    sc = oracle.Scaler(scale, T)
    o = {"p": h["p"].copy(), "m": h["m"].copy(), "v": h["v"].copy(),
         "ew": [e.copy() for e in h["ew"]], "es": [e.copy() for e in h["es"]],
         "plp": h["plp"].copy() if pdtype else None}
    # the GPU's state as it enters a step, on the host (errors explicit)
    gprev = {"m": to_host(d["m"]), "p": to_host(d["p"]),
             "ew": [deferred_error(to_host(d["ew"][i]), float(d["wscale"][i])) for i in range(nd)],
             "es": [deferred_error(to_host(d["es"][j]), float(d["sscale"][j])) for j in range(nd)]}
    for i in range(nd):  # the same start on both sides
        assert gprev["ew"][i].tobytes() == o["ew"][i].tobytes()
        assert gprev["es"][i].tobytes() == o["es"][i].tobytes()
    touched = np.zeros(n, bool)
    flips = 0
    for step in range(steps):
        for i in range(nd):
            h["g"][i] = zs.host_grad(n, 950 + 10 * step + i, step, scale, gdtype)
            d["g"][i] = to_dev(h["g"][i], gdtype)
        o_in = {"m": o["m"].copy(), "p": o["p"].copy(), "ew": [e.copy() for e in o["ew"]],
                "es": [e.copy() for e in o["es"]]}
        run_gpu_step(zp, d, nd, S, numel, zhp, T, pdtype)
        res = oracle.onebit_step(h["g"], gdtype, S, numel, o["p"], o["m"], o["v"], o["ew"], o["es"],
                                 o["plp"], pdtype or "f16", hp, sc, T)
        so = res.step.scalars
        gst = zp.parse_state(d["state"][0])
        assert not res.step.skip and not gst["last_skipped"] and gst["step"] == sc.step
        assert abs(gst["last_norm"] - res.step.norm) <= 1e-6 * res.step.norm
        clip_o, clip_g = np.float32(so["clip"]), np.float32(gst["last_clip"])
        b1, omb1 = float(so["beta1"]), float(so["one_minus_beta1"])
        dm_in = np.abs(gprev["m"].astype(np.float64) - o_in["m"])
        # ---- workers
        gw, ow = d["wscale"].cpu().numpy().astype(np.float64), np.array(res.worker_scales, np.float64)
        wflip = []
        for i in range(nd):
            gu = _abs(oracle.from_lp(h["g"][i], gdtype) if gdtype != "f32" else h["g"][i]) * so["inv_scale"]
            dg = gu * abs(float(clip_g) - float(clip_o))
            if clip_g != clip_o:
                dg += 2 * U * gu * max(float(clip_g), float(clip_o))
            de_in = np.abs(gprev["ew"][i].astype(np.float64) - o_in["ew"][i])
            x_o, x_g = res.worker_x[i], to_host(d["ew"][i])
            diff_in = (dm_in > 0) | (de_in > 0) | (dg > 0)
            bx = b1 * dm_in + omb1 * dg + de_in
            bx = bx * (1 + 4 * U) + np.where(
                diff_in, 8 * U * (b1 * _abs(o_in["m"]) + omb1 * gu * float(clip_o) + _abs(o_in["ew"][i])
                                  + _abs(x_o)) + TINY, 0.0)
            dx = np.abs(x_g.astype(np.float64) - x_o)
            assert np.all(dx <= bx), f"step {step} worker {i}: x beyond its bound"
            bs = np.sqrt(np.sum(bx * bx) / n) * (1 + U) + 2.0 ** -22 * ow[i]
            assert abs(gw[i] - ow[i]) <= bs, f"step {step} worker {i}: scale {gw[i]!r} oracle {ow[i]!r}"
            flip = (x_g < 0) != (x_o < 0)
            assert np.all(_abs(x_o[flip]) <= bx[flip]), f"step {step} worker {i}: a sign flipped beyond its bound"
            wflip.append(flip)
            flips += int(flip.sum())
            touched |= flip
            e_g = deferred_error(x_g, gw[i])
            ds = np.where(flip, gw[i] + ow[i], abs(gw[i] - ow[i]))
            be = dx + ds + np.where((dx > 0) | (ds > 0), 4 * U * (_abs(o["ew"][i]) + _abs(x_o)) + TINY, 0.0)
            assert np.all(np.abs(e_g.astype(np.float64) - o["ew"][i]) <= be), f"step {step} worker {i}: error"
            gprev["ew"][i] = e_g
        # ---- servers
        gsv, osv = d["sscale"].cpu().numpy().astype(np.float64), np.array(res.server_scales, np.float64)
        m_all = to_host(d["m"]).astype(np.float64)
        for j in range(nd):
            seg = slice(j * S, (j + 1) * S)
            dc = sum(np.where(wflip[i][seg], gw[i] + ow[i], abs(gw[i] - ow[i])) for i in range(nd))
            df_in = np.abs(gprev["es"][j].astype(np.float64) - o_in["es"][j])
            y_o, y_g = res.server_x[j], to_host(d["es"][j])
            diff_in = (dc > 0) | (df_in > 0)
            by = dc / nd + df_in
            # roundings: the rank-order sum (Nd - 1 additions, each within
            # u of a partial sum <= the sum of the scales), the mean, y
            by = by * (1 + 4 * U) + np.where(
                diff_in, 4 * U * (ow.sum() + _abs(y_o) + _abs(o_in["es"][j])) + TINY, 0.0)
            dy = np.abs(y_g.astype(np.float64) - y_o)
            assert np.all(dy <= by), f"step {step} server {j}: y beyond its bound"
            bt = np.sqrt(np.sum(by * by) / S) * (1 + U) + 2.0 ** -20 * osv[j]
            assert abs(gsv[j] - osv[j]) <= bt, f"step {step} server {j}: scale {gsv[j]!r} oracle {osv[j]!r}"
            flip = (y_g < 0) != (y_o < 0)
            assert np.all(_abs(y_o[flip]) <= by[flip]), f"step {step} server {j}: a sign flipped beyond its bound"
            flips += int(flip.sum())
            touched[seg] |= flip
            f_g = deferred_error(y_g, gsv[j])
            dt = np.where(flip, gsv[j] + osv[j], abs(gsv[j] - osv[j]))
            bf = dy + dt + np.where((dy > 0) | (dt > 0), 4 * U * (_abs(o["es"][j]) + _abs(y_o)) + TINY, 0.0)
            assert np.all(np.abs(f_g.astype(np.float64) - o["es"][j]) <= bf), f"step {step} server {j}: error"
            gprev["es"][j] = f_g
            # ---- the synchronised momentum of this chunk: +-t exactly
            assert np.all(np.abs(m_all[seg] - o["m"][seg]) <= dt), f"step {step} chunk {j}: momentum"
        # ---- the update with the frozen variance
        p_g = to_host(d["p"])
        dm = np.abs(m_all - o["m"])[:numel]
        dp_in = np.abs(gprev["p"].astype(np.float64) - o_in["p"])[:numel]
        den = np.sqrt(_abs(o["v"][:numel])) * float(so["inv_sqrt_bc2"]) + float(so["eps"])
        st_sz, lrwd = float(so["step_size"]), float(so["lr_wd"])
        bp = dp_in * (1 + lrwd) + st_sz * dm / den * (1 + 4 * U)
        bp += np.where((dp_in > 0) | (dm > 0), 8 * U * (_abs(o["p"][:numel]) + st_sz * _abs(o["m"][:numel]) / den
                                                        + lrwd * _abs(o_in["p"][:numel])) + TINY, 0.0)
        assert np.all(np.abs(p_g[:numel].astype(np.float64) - o["p"][:numel]) <= bp), f"step {step}: master"
        if pdtype:
            assert np.array_equal(to_host(d["plp"])[:numel], oracle.to_lp(p_g[:numel], pdtype)), \
                f"step {step}: the low-precision copy is not the GPU master rounded"
        gprev["m"], gprev["p"] = to_host(d["m"]), p_g
    # flips are rare events at the edge of zero, not a systematic difference
    assert flips <= max(4, n // 1000), flips
    assert touched.sum() <= flips


@pytest.mark.parametrize("nd,S", [(2, 4096)])
def test_onebit_step_with_huge_momentum(zp, nd, S):
    """Momentum values near 1e21 make the worker's and the server's squares
    overflow binary32 (binary64 takes over for those vectors): the scales
    stay finite and within the summation-order bound of the oracle's, and
    the step is the oracle's bit for bit once handed the GPU's scales."""
    T = 70
    h, d = setup(zp, nd, S, "f16", "f16", 4321, 1024.0, T)
    n = nd * S
    rng = np.random.default_rng(11)
    big = rng.choice(n, 40, replace=False)
    h["m"][big] = (np.where(rng.random(40) < 0.5, -1.0, 1.0) * rng.uniform(1.0, 2.0, 40) * 1e21).astype(np.float32)
    d["m"].copy_(torch.from_numpy(h["m"]))
    run_gpu_step(zp, d, nd, S, n, zp.HParams(), T, "f16")
    gw = d["wscale"].cpu().numpy()
    assert np.all(np.isfinite(gw)) and np.all(gw > 1e18)
    check_step(zp, h, d, nd, S, n, "f16", "f16", oracle.HParams(), oracle.Scaler(1024.0, T), T)


@pytest.mark.parametrize("nd,S", [(1, 1024), (4, 8192), (16, 2048)])
def test_onebit_compressed_momentum(zp, nd, S):
    """Step 1 from the dense warm-up momentum; steps 2 and 3 read the
    momentum as the previous servers' signs and scales (the update writes no
    dense m): the same results as the oracle's dense momentum, which after a
    compression step is exactly +-scale."""
    T = 60
    h, d = setup(zp, nd, S, "f16", "f16", 300 + nd, 1024.0, T)
    n = nd * S
    hp, zhp = oracle.HParams(), zp.HParams()
    sc = oracle.Scaler(1024.0, T)
    for step in range(3):
        for i in range(nd):
            h["g"][i] = zs.host_grad(n, 700 + 10 * step + i, step, 1024.0, "f16")
            d["g"][i] = to_dev(h["g"][i], "f16")
        run_gpu_step(zp, d, nd, S, n - 5, zhp, T, "f16", compressed=step > 0)
        check_step(zp, h, d, nd, S, n - 5, "f16", "f16", hp, sc, T, dense_m=step == 0)
    # the compressed momentum the GPU holds is the oracle's dense one
    sb, ss = words(d["sbits"]), d["sscale"].cpu().numpy()
    idx = np.arange(n)
    dense = np.where(bit_at(sb, idx) == 1, ss[idx // S], -ss[idx // S]).astype(np.float32)
    assert dense.tobytes() == h["m"].tobytes()


def test_onebit_overflow_skips_everything(zp):
    nd, S, T = 2, 2048, 30
    h, d = setup(zp, nd, S, "f16", "f16", 5, 4096.0, T, inf_at=(1, 777))
    before = {k: [to_host(t).tobytes() for t in (d[k] if isinstance(d[k], list) else [d[k]])]
              for k in ("p", "m", "ew", "es", "plp", "wscale", "sscale", "wbits", "sbits")}
    run_gpu_step(zp, d, nd, S, nd * S, zp.HParams(), T, "f16")
    for k, v in before.items():
        assert [to_host(t).tobytes() for t in (d[k] if isinstance(d[k], list) else [d[k]])] == v, k
    st = zp.parse_state(d["state"][0])
    assert st["last_skipped"] == 1 and st["step"] == T and st["loss_scale"] == 2048.0


def test_onebit_full_size_rank0_sampled(zp):
    """The benchmark's call sequence at full size (GPT-2 1.5B, Nd = 16,
    rank 0): the worker over all 1,557,612,544 elements, the server on
    chunk 0 with the other workers' signs and scales as received messages,
    and the update; sampled elements against the oracle (with the GPU's
    scales) and the scales against the norm property ||x||_2 = scale *
    sqrt(n) evaluated in binary64 on the device."""
    numel_list = zs.WORKLOADS["gpt2_1p5b_nd16"]["numel"]()
    nd = 16
    lay = zp.zero_partition_layout(numel_list, nd, 128)
    S, numel = lay.shard_numel, sum(numel_list)
    n = nd * S
    dev = torch.device("cuda")
    g = torch.empty(n, dtype=torch.float16, device=dev)
    zs.device_grad_into(g, 31, 0, 65536.0)
    m = zs.device_normal(n, 1e-3, 32, "misc", 1)
    # the worker's error; with its scale 0 the deferred form is the error itself
    e = zs.device_normal(n, 1e-4, 32, "misc", 2)
    v = zs.device_normal(n, 1e-3, 32, "misc", 3).square_()
    p = zs.device_normal(n, 0.02, 32, "master")
    plp = p.half()
    idx = zs.sample_indices(n, 200_000, 5)
    ti = torch.from_numpy(idx).to(dev)
    h_g, h_m, h_e = to_host(g[ti]), to_host(m[ti]), to_host(e[ti])
    h_p, h_v = to_host(p[ti]), to_host(v[ti])
    state = state_at(zp, 65536.0, 1000)
    ws = zp.new_workspace(1, n)
    zp.zero_grad_norm_overflow(g, state, ws)
    bits = torch.zeros(n // 32, dtype=torch.int32, device=dev)
    wscale = torch.zeros(nd, dtype=torch.float32, device=dev)
    hp = zp.HParams()
    zp.zero_onebit_worker(g, m, e, bits, wscale[0:1], hp, 1000, state, ws)
    torch.cuda.synchronize()
    # the norm property, in binary64 on the device, over the compressed
    # value x the array now holds; and every sign bit is the sign of x
    sc0 = float(wscale[0])
    shifts = torch.arange(32, device=dev, dtype=torch.int32)
    tot = 0.0
    for s0 in range(0, n, 1 << 27):
        s1 = min(n, s0 + (1 << 27))
        plus = ((bits[s0 // 32:s1 // 32].view(-1, 1) >> shifts) & 1).reshape(-1).bool()
        x = e[s0:s1].double()
        assert torch.equal(plus, ~(x < 0)), f"signs of [{s0}, {s1})"
        tot += float((x * x).sum())
    norm = (tot / n) ** 0.5
    assert abs(sc0 - norm) <= SCALE_REL * norm
    # sampled elements, with the GPU's scale
    hp_o = oracle.HParams()
    st = oracle.frozen_variance(oracle.decide(hp_o, oracle.Scaler(65536.0, 1000), 0.0, 0), hp_o, 1000)
    xo = np.empty(idx.size, np.float32)
    ob, _ = oracle.onebit_worker(h_g, "f16", st, h_m, h_e, scale=sc0, x_out=xo)
    w_all = words(bits)
    assert np.array_equal(bit_at(w_all, idx), bit_at(ob, np.arange(idx.size)))
    assert to_host(e[ti]).tobytes() == xo.tobytes()
    assert deferred_error(to_host(e[ti]), sc0).tobytes() == h_e.tobytes()
    # server on chunk 0: the other workers' signs and scales are messages
    gen = torch.Generator(device=dev)
    gen.manual_seed(zs.stream_seed(0, "misc", 9))
    others = [torch.randint(-2 ** 31, 2 ** 31 - 1, (S // 32,), dtype=torch.int32, device=dev, generator=gen)
              for _ in range(nd - 1)]
    wscale[1:] = torch.rand(nd - 1, device=dev, generator=gen) * 1e-3 + 1e-4
    es = zs.device_normal(S, 1e-4, 33, "misc", 4)
    sbits = torch.randint(-2 ** 31, 2 ** 31 - 1, (n // 32,), dtype=torch.int32, device=dev, generator=gen)
    sscale = torch.rand(nd, device=dev, generator=gen) * 1e-3 + 1e-4
    sidx = zs.sample_indices(S, 50_000, 6)
    tsi = torch.from_numpy(sidx).to(dev)
    # the server's error in deferred form: es and its previous scale sscale[0]
    f = deferred_error(to_host(es[tsi]), float(sscale[0]))
    f = np.concatenate([f, np.zeros((-sidx.size) % 32, np.float32)])
    chunk_words = [w_all[:S // 32]] + [words(o) for o in others]
    sub = [pack(bit_at(w, sidx)) for w in chunk_words]
    zp.zero_onebit_server([bits[:S // 32]] + others, wscale, es, sbits[:S // 32], sscale[0:1], ws)
    torch.cuda.synchronize()
    s0 = float(sscale[0])
    xo = np.empty(f.size, np.float32)
    ob, _ = oracle.onebit_server(sub, list(wscale.cpu().numpy()), f, scale=s0, x_out=xo)
    assert to_host(es[tsi]).tobytes() == xo[:sidx.size].tobytes()
    assert np.array_equal(bit_at(words(sbits[:S // 32]), sidx), bit_at(ob, np.arange(sidx.size)))
    # the update; the other chunks' signs and scales are messages
    tail_p = to_host(p[numel:]).copy()
    zp.zero_onebit_update(sbits, sscale, S, numel, p, m, v, plp, ws)
    torch.cuda.synchronize()
    keep = idx < numel
    uidx = idx[keep]
    tu = torch.from_numpy(uidx).to(dev)
    hp_s, hv_s = h_p[keep].copy(), h_v[keep].copy()
    hm_s = np.zeros_like(hp_s)
    per_scale = sscale.cpu().numpy()[uidx // S]
    # S = 1: each sampled element is its own chunk with its own scale
    oracle.onebit_update(pack(bit_at(words(sbits), uidx)), list(per_scale), 1, uidx.size, hp_s, hm_s, hv_s,
                         None, "f16", st)
    assert to_host(p[tu]).tobytes() == hp_s.tobytes()
    assert to_host(m[tu]).tobytes() == hm_s.tobytes()
    assert np.array_equal(to_host(plp[tu]), oracle.to_lp(hp_s, "f16"))
    # the padding past numel is not parameters: untouched; the momentum
    # covers the whole padded buffer
    assert to_host(p[numel:]).tobytes() == tail_p.tobytes()
    tail = np.arange(numel, n)
    sw, ss = words(sbits), sscale.cpu().numpy()
    want_m = np.where(bit_at(sw, tail) == 1, ss[tail // S], -ss[tail // S]).astype(np.float32)
    assert to_host(m[numel:]).tobytes() == want_m.tobytes()


def test_onebit_argument_errors(zp):
    dev = "cuda"
    g = torch.zeros(100, dtype=torch.float16, device=dev)  # not a multiple of 32
    f = torch.zeros(100, device=dev)
    bits = torch.zeros(3, dtype=torch.int32, device=dev)
    st, ws = state_at(zp, 1.0, 5), zp.new_workspace(1, 128)
    with pytest.raises(zp.ZeroError) as e:
        zp.zero_onebit_worker(g, f, f.clone(), bits, torch.zeros(1, device=dev), zp.HParams(), 5, st, ws)
    assert e.value.code == -4
    g = torch.zeros(128, dtype=torch.float16, device=dev)
    f = torch.zeros(128, device=dev)
    bits = torch.zeros(4, dtype=torch.int32, device=dev)
    with pytest.raises(zp.ZeroError) as e:  # freeze step must be a step count
        zp.zero_onebit_worker(g, f, f.clone(), bits, torch.zeros(1, device=dev), zp.HParams(), 0, st, ws)
    assert e.value.code == -1
    big = torch.zeros(256, device=dev)
    with pytest.raises(zp.ZeroError) as e:  # numel past nd * S
        zp.zero_onebit_update(bits, torch.ones(1, device=dev), 128, 129, big, None, big.clone(), None, ws)
    assert e.value.code == -4


def server_case(zp, nd, S, seed, T=10):
    """Random worker signs and scales and a server error for one chunk, with
    the step's decision (no overflow) taken in the workspace by a worker call
    on 32 elements."""
    rng = np.random.default_rng(seed)
    w = S // 32
    hb = [rng.integers(0, 2 ** 32, w, dtype=np.uint64).astype(np.uint32) for _ in range(nd)]
    hs = rng.uniform(1e-4, 1.1e-3, nd).astype(np.float32)
    hf = (rng.standard_normal(S) * 1e-4).astype(np.float32)
    d = {
        "wbits": [torch.from_numpy(b.view(np.int32)).cuda() for b in hb],
        "wscale": torch.from_numpy(hs).cuda(),
        "es": torch.from_numpy(hf.copy()).cuda(),
        "bits": torch.zeros(w, dtype=torch.int32, device="cuda"),
        "scale": torch.zeros(1, dtype=torch.float32, device="cuda"),
        "state": state_at(zp, 1024.0, T),
        "ws": zp.new_workspace(nd, nd * S),
    }
    z = torch.zeros(32, dtype=torch.float32, device="cuda")
    zp.zero_onebit_worker(torch.zeros(32, dtype=torch.float16, device="cuda"), z, z.clone(),
                          torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.zeros(1, dtype=torch.float32, device="cuda"), zp.HParams(), T,
                          d["state"], d["ws"])
    return hb, hs, hf, d


def check_server(hb, hs, hf, d):
    """The GPU's server pass against the oracle's (handed the GPU's scale):
    the compressed value, the error it stands for and the signs bit for
    bit, the scale within the norm's summation-order bound.  The server
    started from scale 0, so its array was the explicit error hf."""
    torch.cuda.synchronize()
    gs = float(d["scale"][0])
    _, free = oracle.onebit_server([b.copy() for b in hb], list(hs), hf.copy())
    assert abs(gs - free) <= 4 * SCALE_REL * free, "server scale"
    f = hf.copy()
    x = np.empty_like(f)
    ob, _ = oracle.onebit_server(hb, list(hs), f, scale=gs, x_out=x)
    assert to_host(d["es"]).tobytes() == x.tobytes(), "server compressed value"
    assert deferred_error(x, gs).tobytes() == f.tobytes(), "server error"
    assert np.array_equal(words(d["bits"]), ob), "server signs"


@pytest.mark.parametrize("nd,S", [(1, 1184), (5, 4128), (8, 1184), (9, 4128), (14, 8192), (15, 4128),
                                  (16, 1_280_000), (17, 4128), (24, 1184), (33, 8192), (256, 4128),
                                  (257, 1184), (300, 4128)])
def test_onebit_server_worker_counts(zp, nd, S):
    """The server pass over every split of its sum: the tabulated first
    min(nd, 14) workers, workers 14 and 15 added after the table, whole and
    partial groups of 8 past 16; power-of-two counts (the mean as a product)
    and others (a division); pointers as a launch argument (nd <= 256) and
    as a workspace table; chunks that end inside a warp's 1024 elements."""
    hb, hs, hf, d = server_case(zp, nd, S, 1000 + nd)
    zp.zero_onebit_server(d["wbits"], d["wscale"], d["es"], d["bits"], d["scale"], d["ws"])
    check_server(hb, hs, hf, d)


def test_onebit_server_equal_scales(zp):
    """Equal worker scales and a zero server error: the table holds many
    equal entries and every element with as many + as - signs sums to an
    exact zero (the mean's zero numerator takes the division's special
    path on other counts; here the product)."""
    nd, S = 16, 8192
    hb, hs, hf, d = server_case(zp, nd, S, 4242)
    hs[:] = np.float32(5e-4)
    d["wscale"].copy_(torch.from_numpy(hs))
    hf[:] = 0.0
    d["es"].zero_()
    zp.zero_onebit_server(d["wbits"], d["wscale"], d["es"], d["bits"], d["scale"], d["ws"])
    check_server(hb, hs, hf, d)


def _off16(t):
    """The values of t in a buffer that starts 16 bytes past a 32-byte
    boundary."""
    buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=t.device)
    v = buf[4:]
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


@pytest.mark.parametrize("compressed", [False, True])
def test_onebit_16_byte_aligned_arrays(zp, compressed):
    """fp32 arrays on a 16-byte but not a 32-byte boundary take two 16-byte
    accesses per 8 elements instead of one 32-byte access, in all three
    calls: the same results bit for bit."""
    nd, S, T = 4, 4096, 40
    _, d = setup(zp, nd, S, "f16", "f16", 77, 1024.0, T)
    clone = {k: ([t.clone() for t in v] if isinstance(v, list) else v.clone()) for k, v in d.items()}
    for k in ("ew", "es"):
        clone[k] = [_off16(t) for t in clone[k]]
    for k in ("p", "m", "v"):
        clone[k] = _off16(clone[k])
    for dd in (d, clone):
        run_gpu_step(zp, dd, nd, S, nd * S - 3, zp.HParams(), T, "f16", compressed=compressed)
    for k in ("ew", "es", "wbits", "sbits", "wscale", "sscale", "p", "m", "plp", "state"):
        a = d[k] if isinstance(d[k], list) else [d[k]]
        b = clone[k] if isinstance(clone[k], list) else [clone[k]]
        assert [to_host(t).tobytes() for t in a] == [to_host(t).tobytes() for t in b], k
