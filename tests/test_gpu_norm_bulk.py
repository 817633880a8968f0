"""Pass 1 over flat shards large enough for the shared-memory-staged kernel,
against the oracle.

From 8 whole chunks of 16 KiB per SM on, pass 1 over a flat shard stages the
gradient through shared memory with bulk copies: block b of G (two per SM)
takes the chunks b, b + G, ..., and the last block takes the elements after
the last whole chunk with plain loads.  The sizes below sit on both sides of
that threshold and put the remainder in every shape (none, a scalar tail
only, vectors and a tail, one element short of a chunk); inf and NaN go to
the first element, both sides of a chunk boundary, the last element of the
last whole chunk, the remainder and the tail.  The norm is held to the
oracle's binary64 sum within 1e-6, the overflow flag exactly, whole steps
element by element; no wait in any of these calls gives up."""
import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import NORM_REL, to_dev  # noqa: E402
from test_gpu_parity import run_full  # noqa: E402

EB = {"f16": 2, "bf16": 2, "f32": 4}
CHUNK_BYTES = 16 << 10
CHUNKS_PER_SM = 8
BLOCKS_PER_SM = 2


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def chunk_elems(gdtype):
    return CHUNK_BYTES // EB[gdtype]


def threshold(gdtype):
    """Elements of the smallest flat shard that takes the staged kernel."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return CHUNKS_PER_SM * sms * chunk_elems(gdtype)


SHAPES = {
    "below": lambda t, c: t - 1,            # one chunk short: the register-loaded kernel
    "exact": lambda t, c: t,                # whole chunks only, no remainder
    "tail5": lambda t, c: t + 5,            # a scalar tail only
    "ragged": lambda t, c: 2 * t + 8 * 1001 + 3,  # remainder vectors and a tail
    "almost": lambda t, c: 2 * t + c - 1,   # one element short of another chunk
}


def grad(n, gdtype, seed, scale=1.0, kind=None):
    if kind is not None:
        return zs.host_cast(zs.host_wide_range(n, seed, kind), gdtype)
    return zs.host_grad(n, seed, 0, scale, gdtype)


def norm_of(zp, state):
    st = zp.parse_state(state)
    return st["sumsq"], st["found_inf"]


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("gdtype", ["f16", "bf16", "f32"])
def test_norm_matches_oracle(zp, gdtype, shape):
    n = SHAPES[shape](threshold(gdtype), chunk_elems(gdtype))
    scale = 1024.0 if gdtype == "f16" else 1.0
    g = grad(n, gdtype, 11, scale)
    dg = to_dev(g, gdtype)
    state, ws = zp.new_state(scale), zp.new_workspace(1, n)
    zp.zero_grad_norm_overflow(dg, state, ws)
    sumsq, found = norm_of(zp, state)
    ora, bad = oracle.norm_overflow([g], gdtype, scale)
    assert found == 0.0 and bad == 0
    assert abs(np.sqrt(sumsq) - np.sqrt(ora)) <= NORM_REL * np.sqrt(ora), (sumsq, ora)
    # the same bits on a second run (fixed chunk, thread and reduction order)
    zp.zero_grad_norm_overflow(dg, state, ws)
    assert norm_of(zp, state)[0] == sumsq
    assert zp.zero_workspace_stalls(ws) == 0


def positions(n, gdtype):
    """Overflow positions: around chunk boundaries, the last element of the
    last whole chunk, in the remainder and in the tail."""
    c = chunk_elems(gdtype)
    nch = n // c
    return {
        "first": 0,
        "chunk0_last": c - 1,
        "chunk1_first": c,
        "last_whole_chunk": nch * c - 1,
        "remainder": nch * c + 8,
        "tail": n - 1,
    }


@pytest.mark.parametrize("where", ["first", "chunk0_last", "chunk1_first", "last_whole_chunk", "remainder",
                                   "tail"])
@pytest.mark.parametrize("nan", [False, True])
@pytest.mark.parametrize("gdtype", ["f16", "bf16", "f32"])
def test_overflow_positions(zp, gdtype, where, nan):
    n = SHAPES["ragged"](threshold(gdtype), chunk_elems(gdtype))
    pos = positions(n, gdtype)[where]
    g = grad(n, gdtype, 12)
    g[pos] = zs.host_cast(np.array([np.nan if nan else -np.inf], np.float32), gdtype)[0]
    state, ws = zp.new_state(1.0), zp.new_workspace(1, n)
    zp.zero_grad_norm_overflow(to_dev(g, gdtype), state, ws)
    _, found = norm_of(zp, state)
    assert oracle.norm_overflow([g], gdtype, 1.0)[1] == 1
    assert found == 1.0
    assert zp.zero_workspace_stalls(ws) == 0


@pytest.mark.parametrize("gdtype,pdtype", [("f16", "f16"), ("bf16", "bf16"), ("f32", "f16")])
@pytest.mark.parametrize("whole", [True, False], ids=["zero_step", "two_calls"])
def test_steps_against_oracle(zp, gdtype, pdtype, whole):
    """Three steps with clipping on, every element: through zero_step the
    staged kernel's last block also takes the step decision."""
    n = SHAPES["ragged"](threshold(gdtype), chunk_elems(gdtype))
    scale = 4096.0 if gdtype == "f16" else 1.0
    st, skipped = run_full(zp, n, gdtype, pdtype, 3, scale, max_norm=0.5, seed=13, whole=whole)
    assert skipped == 0 and st["step"] == 3


@pytest.mark.parametrize("whole", [True, False], ids=["zero_step", "two_calls"])
def test_overflow_step_skipped_at_a_chunk_boundary(zp, whole):
    """An inf at the first element of block 0's second chunk: the step is
    skipped with the state unchanged and the scale halved."""
    n = SHAPES["ragged"](threshold("f16"), chunk_elems("f16"))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pos = BLOCKS_PER_SM * sms * chunk_elems("f16")
    st, skipped = run_full(zp, n, "f16", "f16", 3, 65536.0, seed=14, inf_step=1, inf_pos=pos, whole=whole)
    assert skipped == 1 and st["step"] == 2 and st["loss_scale"] == 32768.0


@pytest.mark.parametrize("gdtype", ["bf16", "f32"])
@pytest.mark.parametrize("kind", zs.WIDE_KINDS)
def test_norm_over_the_binary32_range(zp, gdtype, kind):
    n = SHAPES["tail5"](threshold(gdtype), chunk_elems(gdtype))
    g = grad(n, gdtype, 15, kind=kind)
    state, ws = zp.new_state(1.0), zp.new_workspace(1, n)
    zp.zero_grad_norm_overflow(to_dev(g, gdtype), state, ws)
    sumsq, found = norm_of(zp, state)
    ora, bad = oracle.norm_overflow([g], gdtype, 1.0)
    assert found == 0.0 and bad == 0 and ora > 0.0
    assert np.isfinite(sumsq)
    assert abs(np.sqrt(sumsq) - np.sqrt(ora)) <= NORM_REL * np.sqrt(ora), (kind, sumsq, ora)


def test_accumulate_folds_two_calls(zp):
    """accumulate = 1 adds the second shard's sum and flag to the first's."""
    n = SHAPES["ragged"](threshold("f16"), chunk_elems("f16"))
    g0, g1 = grad(n, "f16", 16, 512.0), grad(n, "f16", 17, 512.0)
    state, ws = zp.new_state(512.0), zp.new_workspace(1, n)
    zp.zero_grad_norm_overflow(to_dev(g0, "f16"), state, ws)
    zp.zero_grad_norm_overflow(to_dev(g1, "f16"), state, ws, accumulate=True)
    sumsq, found = norm_of(zp, state)
    ora = oracle.norm_overflow([g0], "f16", 512.0)[0] + oracle.norm_overflow([g1], "f16", 512.0)[0]
    assert found == 0.0
    assert abs(np.sqrt(sumsq) - np.sqrt(ora)) <= NORM_REL * np.sqrt(ora)
    assert zp.zero_workspace_stalls(ws) == 0


def test_stalls_argument_errors(zp):
    """NULL arguments, a workspace off its 256-byte boundary and host
    memory are refused on the host."""
    import ctypes
    EINVAL, EALIGN = -1, -2
    ws = zp.new_workspace(1, 16)
    out = ctypes.c_uint32()
    lib = zp.lib()
    assert lib.zero_workspace_stalls(None, ctypes.byref(out), None) == EINVAL
    assert lib.zero_workspace_stalls(ctypes.c_void_p(ws.data_ptr()), None, None) == EINVAL
    assert lib.zero_workspace_stalls(ctypes.c_void_p(ws.data_ptr() + 16), ctypes.byref(out), None) == EALIGN
    host = (ctypes.c_uint8 * 512)()
    addr = (ctypes.addressof(host) + 255) & ~255
    assert lib.zero_workspace_stalls(ctypes.c_void_p(addr), ctypes.byref(out), None) == EINVAL
    assert zp.zero_workspace_stalls(ws) == 0


def test_managed_gradient_is_read_with_ordinary_loads(zp):
    """A gradient in managed memory (cudaMallocManaged) above the staged
    kernel's size: the library never points a bulk copy at memory that may
    have to be faulted in, so pass 1 takes the register-loaded kernel here,
    and the norm is still the oracle's within 1e-6."""
    import ctypes
    from zero_partitioned_mixed_layout_gb300.binding import _TList
    rt = ctypes.CDLL("libcudart.so.13")
    vp = ctypes.c_void_p
    n = SHAPES["ragged"](threshold("f16"), chunk_elems("f16"))
    g = grad(n, "f16", 18, 1024.0)
    dg = vp()
    assert rt.cudaMallocManaged(ctypes.byref(dg), ctypes.c_size_t(g.nbytes), 1) == 0  # attach global
    try:
        assert rt.cudaDeviceSynchronize() == 0
        ctypes.memmove(dg, g.ctypes.data, g.nbytes)
        state, ws = zp.new_state(1024.0), zp.new_workspace(1, n)
        ptrs = (vp * 1)(dg)
        numel = (ctypes.c_int64 * 1)(n)
        tl = _TList(ptrs, numel, 1, 0)
        torch.cuda.synchronize()
        rc = zp.lib().zero_grad_norm_overflow(ctypes.byref(tl), vp(state.data_ptr()), 0, vp(ws.data_ptr()),
                                              ws.numel(), vp(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, zp.zero_strerror(rc)
        torch.cuda.synchronize()
        sumsq, found = norm_of(zp, state)
        ora, bad = oracle.norm_overflow([g], "f16", 1024.0)
        assert found == 0.0 and bad == 0
        assert abs(np.sqrt(sumsq) - np.sqrt(ora)) <= NORM_REL * np.sqrt(ora)
        assert zp.zero_workspace_stalls(ws) == 0
    finally:
        assert rt.cudaFree(dg) == 0


@pytest.mark.parametrize("gdtype", ["f16", "f32"])
def test_many_calls_give_the_same_bits(zp, gdtype):
    """400 calls back to back on one stream over the same gradient: the ring
    of bulk copies and its barriers give the same sum of squares bit for bit
    every time, and no wait gives up."""
    n = SHAPES["almost"](threshold(gdtype), chunk_elems(gdtype))
    g = to_dev(grad(n, gdtype, 19, 1.0), gdtype)
    state, ws = zp.new_state(1.0), zp.new_workspace(1, n)
    sums = torch.empty(400, dtype=torch.float64, device="cuda")
    head = state[:8].view(torch.float64)
    for k in range(400):
        zp.zero_grad_norm_overflow(g, state, ws)
        sums[k] = head[0]
    torch.cuda.synchronize()
    assert torch.unique(sums).numel() == 1 and sums[0].item() > 0
    assert zp.zero_workspace_stalls(ws) == 0
