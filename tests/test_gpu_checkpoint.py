"""Checkpoint / resume and guard bands.

The optimizer's whole state is plain buffers -- the fp32 master, momentum and
variance, the low-precision copy, and the 64-byte zero_state_t (loss scale,
step count, good-step run) -- so a checkpoint is a copy of those and a resume
is a copy back into fresh buffers with a fresh workspace.  A resumed run
equals the uninterrupted one bit for bit, also when the checkpoint is taken
with Nd = 4 shards and resumed with Nd = 2 (re-sharded through the layout).
Guard bands around every array stay untouched by every kernel that writes."""
import math

import numpy as np
import pytest

import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import TORCH, to_dev, to_host  # noqa: E402


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def _raw(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().tobytes()


def _hp(zp, k):
    lr = 1e-3 * min(1.0, (k + 1) / 5) * 0.5 * (1.0 + math.cos(math.pi * k / 20))
    return zp.HParams(lr=lr, max_norm=0.5)


def _grad(n, k, scale, gdtype):
    g = zs.host_grad(n, 123, k, scale, gdtype)
    if k == 4:
        g[n // 3] = zs.host_cast(np.array([np.inf], np.float32), gdtype)[0]
    return g


@pytest.mark.parametrize("gdtype,pdtype", [("f16", "f16"), ("bf16", "bf16")])
def test_checkpoint_resume_is_bit_identical(zp, gdtype, pdtype):
    """20 steps straight through against 9 steps, a checkpoint to host memory,
    and a resume into fresh buffers and a fresh workspace for the other 11
    (learning-rate schedule, clipping, an overflow at step 4; the resumed
    run's first decision finds no cached bias corrections)."""
    n = 200_003
    scale = 1024.0 if gdtype == "f16" else 1.0
    p0 = zs.host_master(n, 9)

    def fresh():
        return dict(p=torch.from_numpy(p0.copy()).cuda(), m=torch.zeros(n, device="cuda"),
                    v=torch.zeros(n, device="cuda"), lp=torch.zeros(n, dtype=TORCH[pdtype], device="cuda"),
                    st=zp.new_state(scale), ws=zp.new_workspace(1, n))

    def steps(d, ks):
        for k in ks:
            g = to_dev(_grad(n, k, zp.parse_state(d["st"])["loss_scale"], gdtype), gdtype)
            zp.zero_step(g, d["p"], d["m"], d["v"], d["lp"], _hp(zp, k), d["st"], d["ws"])
        torch.cuda.synchronize()

    a = fresh()
    steps(a, range(20))
    b = fresh()
    steps(b, range(9))
    ckpt = {key: b[key].cpu().clone() for key in ("p", "m", "v", "lp", "st")}
    del b
    c = fresh()
    for key in ("p", "m", "v", "lp", "st"):
        c[key].copy_(ckpt[key])
    steps(c, range(9, 20))
    for key in ("p", "m", "v", "lp", "st"):
        assert _raw(a[key]) == _raw(c[key]), key
    st = zp.parse_state(c["st"])
    assert st["step"] == 19 and st["skipped"] == 1


def test_reshard_checkpoint_nd4_to_nd2(zp):
    """Three steps with Nd = 4 emulated ranks (own shard, state and
    workspace; the ranks' 16-byte partials summed between the passes), a
    checkpoint gathered into the flat buffer, then three steps with Nd = 2
    shards cut from it by the Nd = 2 layout: equal bit for bit to six steps
    of the unpartitioned state (clipping off: partition invariance is exact)."""
    numel = [1000, 37, 70_001, 5, 4096, 123_457, 1]
    total = sum(numel)
    scale = 1024.0
    hp = zp.HParams(max_norm=0.0)
    p_flat = zs.host_master(total, 17)

    def grad_flat(k):
        return zs.host_grad(total, 31, k, scale, "f16")

    def run_ranks(nd, p_real, m_real, v_real, lp_real, st_bytes, ks):
        lay = zp.zero_partition_layout(numel, nd, 128)
        S, N = lay.shard_numel, lay.padded_total

        def pad(x, dtype):
            out = np.zeros(N, dtype)
            out[:total] = x
            return out
        fp, fm, fv = pad(p_real, np.float32), pad(m_real, np.float32), pad(v_real, np.float32)
        flp = pad(lp_real, np.uint16)
        ranks = []
        for r in range(nd):
            sl = slice(r * S, (r + 1) * S)
            st = torch.from_numpy(np.frombuffer(st_bytes, np.uint8).copy()).cuda()
            ranks.append(dict(p=to_dev(fp[sl].copy(), "f32"), m=to_dev(fm[sl].copy(), "f32"),
                              v=to_dev(fv[sl].copy(), "f32"),
                              lp=torch.from_numpy(flp[sl].view(np.float16).copy()).cuda(),
                              st=st, ws=zp.new_workspace(1, S)))
        for k in ks:
            g = np.zeros(N, np.float16)
            g[:total] = grad_flat(k)
            gs = [torch.from_numpy(g[r * S:(r + 1) * S].copy()).cuda() for r in range(nd)]
            for r in range(nd):
                zp.zero_grad_norm_overflow(gs[r], ranks[r]["st"], ranks[r]["ws"])
            partial = sum(rk["st"][:16].view(torch.float64) for rk in ranks)
            for rk in ranks:
                rk["st"][:16] = partial.view(torch.uint8)
            for r in range(nd):
                rk = ranks[r]
                zp.zero_adam_step(gs[r], rk["p"], rk["m"], rk["v"], rk["lp"], hp, rk["st"], rk["ws"])
        torch.cuda.synchronize()
        cat = {key: np.concatenate([to_host(rk[key]) for rk in ranks]) for key in ("p", "m", "v", "lp")}
        states = [rk["st"].cpu().numpy().tobytes() for rk in ranks]
        assert all(s == states[0] for s in states)
        for key in ("p", "m", "v"):
            assert not cat[key][total:].any(), f"padding of {key} written"
        return {key: cat[key][:total].copy() for key in cat}, states[0]

    st0 = zp.new_state(scale).cpu().numpy().tobytes()
    z32, z16 = np.zeros(total, np.float32), np.zeros(total, np.uint16)
    # the unpartitioned reference: Nd = 1, six steps
    ref, ref_st = run_ranks(1, p_flat, z32, z32, z16, st0, range(6))
    # Nd = 4 for three steps, then the checkpoint re-sharded to Nd = 2
    mid, mid_st = run_ranks(4, p_flat, z32, z32, z16, st0, range(3))
    out, out_st = run_ranks(2, mid["p"], mid["m"], mid["v"], mid["lp"], mid_st, range(3, 6))
    for key in ("p", "m", "v", "lp"):
        assert out[key].tobytes() == ref[key].tobytes(), key
    # loss scale, step, good steps, skipped; last clip and skip (the last
    # norm's binary64 sum is grouped differently on each partitioning)
    assert out_st[16:48] == ref_st[16:48] and out_st[56:] == ref_st[56:]


GUARD = 64  # elements on each side


def _guarded(n, dtype):
    """A device array of n elements inside a buffer with GUARD sentinel
    elements on each side (the array starts on a 16-byte boundary)."""
    t = TORCH[dtype]
    buf = torch.empty(n + 2 * GUARD, dtype=t, device="cuda")
    bits = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}[t]
    buf.view(bits).fill_(0x7FC05555 if t == torch.float32 else 0x7E55)
    return buf, buf[GUARD:GUARD + n]


def _guards_intact(buf, n):
    t = buf.dtype
    bits = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}[t]
    want = 0x7FC05555 if t == torch.float32 else 0x7E55
    raw = buf.view(bits)
    return bool((raw[:GUARD] == want).all()) and bool((raw[GUARD + n:] == want).all())


@pytest.mark.parametrize("sizes", [[1], [7], [9], [2049], [100_003], [3, 4099, 70_001, 1]])
def test_guard_bands_untouched(zp, sizes):
    """Every array of a step (flat or list), of the fused accumulation and of
    the stage-2 reduction sits between sentinel guard bands: after the calls
    the guards hold their sentinels, for sizes below, at and past a vector and
    a tile."""
    scale = 1024.0
    hp = zp.HParams(max_norm=0.5)
    arrays = []
    lists = {key: [] for key in ("g", "p", "m", "v", "lp")}
    for n in sizes:
        for key, dt in (("g", "f16"), ("p", "f32"), ("m", "f32"), ("v", "f32"), ("lp", "f16")):
            buf, arr = _guarded(n, dt)
            if key == "g":
                arr.copy_(to_dev(zs.host_grad(n, 3, 0, scale, "f16"), "f16"))
            elif key == "p":
                arr.copy_(torch.from_numpy(zs.host_master(n, 3)).cuda())
            else:
                arr.zero_()
            arrays.append((buf, n))
            lists[key].append(arr)
    st = zp.new_state(scale)
    ws = zp.new_workspace(len(sizes), sum(sizes))
    g = lists["g"] if len(sizes) > 1 else lists["g"][0]
    args = [lists[key] if len(sizes) > 1 else lists[key][0] for key in ("p", "m", "v", "lp")]
    for _ in range(2):
        zp.zero_step(g, *args, hp, st, ws)
    # the fused accumulation and the stage-2 reduction on the last size
    n = sizes[-1]
    acc_buf, acc = _guarded(n, "f32")
    mb = []
    for j in range(4):
        b, a = _guarded(n, "bf16")
        a.copy_(to_dev(zs.host_grad(n, 5, 0, 1.0, "bf16", micro=j), "bf16"))
        mb.append((b, a))
    st2 = zp.new_state(1.0)
    ws2 = zp.new_workspace(1, n)
    zp.zero_accumulate_grads_norm(acc, [a for _, a in mb], st2, ws2, True)
    out_buf, out = _guarded(n, "f16")
    reps = []
    for j in range(3):
        b, a = _guarded(n, "f16")
        a.copy_(to_dev(zs.host_grad(n, 6, 0, scale, "f16", micro=j), "f16"))
        reps.append((b, a))
    zp.zero_reduce_grads([a for _, a in reps], out, zp.new_state(scale), ws2)
    torch.cuda.synchronize()
    for buf, n_ in arrays:
        assert _guards_intact(buf, n_), "a step wrote outside its arrays"
    assert _guards_intact(acc_buf, n), "the accumulation wrote outside acc"
    assert _guards_intact(out_buf, n), "the reduction wrote outside out"
    for b, _ in mb + reps:
        assert _guards_intact(b, n), "an input array was written"
