"""zero_grad_norm_overflow_static: pass 1 for callers that cannot allocate
device memory (and so cannot pass a workspace), with its scratch in a static
device array inside the library.  Called through the C ABI and checked,
two calls in a row, against zero_grad_norm_overflow on the same gradients
and against the oracle's binary64 sum on host copies of them, within the
norm tolerance the parity tests use (1e-6 relative); the accumulate mode's
folded sum against the oracle's sum over both calls' arrays."""
import ctypes

import numpy as np
import pytest

import oracle
import zero_synth as zs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gpu_common import to_dev  # noqa: E402

NORM_REL = 1e-6


@pytest.fixture(scope="module")
def zp():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    from zero_partitioned_mixed_layout_gb300.binding import _TList
    so = zp.lib()
    so.zero_grad_norm_overflow_static.argtypes = [ctypes.POINTER(_TList), ctypes.c_void_p,
                                                  ctypes.c_int32, ctypes.c_void_p]
    so.zero_grad_norm_overflow_static.restype = ctypes.c_int
    return zp


def call_static(zp, arrays, state, accumulate=0):
    """The raw C call: grads as a zero_tlist_t, state, accumulate, stream."""
    from zero_partitioned_mixed_layout_gb300.binding import _TList
    n = len(arrays)
    ptrs = (ctypes.c_void_p * n)(*[a.data_ptr() for a in arrays])
    numel = (ctypes.c_int64 * n)(*[a.numel() for a in arrays])
    code = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}[arrays[0].dtype]
    tl = _TList(ptrs, numel, n, code)
    return zp.lib().zero_grad_norm_overflow_static(
        ctypes.byref(tl), ctypes.c_void_p(state.data_ptr()), accumulate,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def head(zp, state):
    st = zp.parse_state(state)
    return st["sumsq"], st["found_inf"]


def host_grads(sizes, dtype, scale, seed):
    return [zs.host_grad(n, seed, 0, scale, dtype, micro=i) for i, n in enumerate(sizes)]


def close(a, b):
    """Norms within NORM_REL, compared on sums of squares."""
    return b > 0 and abs(np.sqrt(a) - np.sqrt(b)) <= NORM_REL * np.sqrt(b)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sizes", [[97_350_784], [5, 70_001, 3, 1 << 20]], ids=["flat", "list"])
def test_static_scratch_matches_workspace_call_and_oracle(zp, dtype, sizes):
    scale = 1024.0 if dtype == "f16" else 1.0
    for call in range(2):  # two calls in a row share the static scratch
        host = host_grads(sizes, dtype, scale, 40 + call)
        arrays = [to_dev(a, dtype) for a in host]
        ref_state, st_state = zp.new_state(scale), zp.new_state(scale)
        ws = zp.new_workspace(len(arrays), sum(sizes))
        zp.zero_grad_norm_overflow(arrays, ref_state, ws)
        rc = call_static(zp, arrays, st_state)
        assert rc == 0, zp.zero_strerror(rc)
        torch.cuda.synchronize()
        (s_ref, f_ref), (s_st, f_st) = head(zp, ref_state), head(zp, st_state)
        s_ora, f_ora = oracle.norm_overflow(host, dtype, scale)
        assert f_st == f_ref == 0.0 and f_ora == 0
        assert close(s_st, s_ref), (s_st, s_ref)
        assert close(s_st, s_ora), (s_st, s_ora)
    # accumulate mode folds a second call into the first: the oracle's sum
    # over both calls' arrays; an overflow in a third call is counted
    first, second = host_grads(sizes, dtype, scale, 50), host_grads(sizes, dtype, scale, 51)
    st_state = zp.new_state(scale)
    assert call_static(zp, [to_dev(a, dtype) for a in first], st_state, 0) == 0
    assert call_static(zp, [to_dev(a, dtype) for a in second], st_state, 1) == 0
    torch.cuda.synchronize()
    s_ora, f_ora = oracle.norm_overflow(first + second, dtype, scale)
    s_st, f_st = head(zp, st_state)
    assert f_st == 0.0 and f_ora == 0 and close(s_st, s_ora), (s_st, s_ora)
    third = [to_dev(a, dtype) for a in host_grads(sizes, dtype, scale, 52)]
    third[-1][-1] = float("inf")
    assert call_static(zp, third, st_state, 1) == 0
    torch.cuda.synchronize()
    assert head(zp, st_state)[1] == 1.0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("kind", zs.WIDE_KINDS)
def test_static_scratch_over_the_binary32_range(zp, dtype, kind):
    """Magnitudes across the binary32 range (values near 1e20, tiny,
    subnormal, near the maximum): the norm within 1e-6 of the oracle's."""
    host = [zs.host_cast(zs.host_wide_range(n, 90 + i, kind), dtype) for i, n in enumerate([100_003, 77])]
    state = zp.new_state(1.0)
    assert call_static(zp, [to_dev(a, dtype) for a in host], state) == 0
    torch.cuda.synchronize()
    s_st, f_st = head(zp, state)
    s_ora, f_ora = oracle.norm_overflow(host, dtype, 1.0)
    assert f_st == 0.0 and f_ora == 0 and close(s_st, s_ora), (kind, s_st, s_ora)


def test_static_scratch_rejects_long_lists(zp):
    arrays = [torch.ones(16, dtype=torch.float16, device="cuda") for _ in range(33)]
    state = zp.new_state(1.0)
    before = state.clone()
    assert call_static(zp, arrays, state) == -6  # ZERO_ECAPACITY: more than 32 arrays
    torch.cuda.synchronize()
    assert torch.equal(before, state), "a rejected call changed the state"
    assert call_static(zp, arrays[:32], state) == 0
    torch.cuda.synchronize()
    assert head(zp, state) == (32 * 16.0, 0.0)


_RESET_SCRIPT = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import zero_partitioned_mixed_layout_gb300 as zp
from zero_partitioned_mixed_layout_gb300.binding import _TList
so = zp.lib()
rt = ctypes.CDLL("libcudart.so.13")
vp = ctypes.c_void_p
so.zero_grad_norm_overflow_static.argtypes = [ctypes.POINTER(_TList), vp, ctypes.c_int32, vp]
so.zero_grad_norm_overflow_static.restype = ctypes.c_int
rng = np.random.default_rng(7)
g = (rng.standard_normal(100_003) * 1e-3).astype(np.float16)
init = zp.zero_state_init(1.0)

def run():
    dg, ds = vp(), vp()
    assert rt.cudaMalloc(ctypes.byref(dg), ctypes.c_size_t(g.nbytes)) == 0
    assert rt.cudaMalloc(ctypes.byref(ds), ctypes.c_size_t(64)) == 0
    assert rt.cudaMemcpy(dg, g.ctypes.data_as(vp), ctypes.c_size_t(g.nbytes), 1) == 0
    assert rt.cudaMemcpy(ds, ctypes.c_char_p(init), ctypes.c_size_t(64), 1) == 0
    ptrs = (vp * 1)(dg)
    numel = (ctypes.c_int64 * 1)(g.size)
    rc = so.zero_grad_norm_overflow_static(ctypes.byref(_TList(ptrs, numel, 1, 0)), ds, 0, None)
    assert rc == 0, zp.zero_strerror(rc)
    out = ctypes.create_string_buffer(64)
    assert rt.cudaMemcpy(out, ds, ctypes.c_size_t(64), 2) == 0
    assert rt.cudaFree(dg) == 0 and rt.cudaFree(ds) == 0
    return zp.parse_state(out.raw)["sumsq"]

first = run()
assert rt.cudaDeviceReset() == 0
second = run()
print(first, second)
assert first == second and first > 0
'''


def test_static_scratch_after_a_device_reset(zp, tmp_path):
    """A device reset replaces the context and the library's module with it:
    the first call after it looks the scratch address up again.  In a child
    process with the CUDA runtime alone (a reset would invalidate this
    process's tensors): the same gradient gives the same sum of squares
    before and after the reset."""
    import os
    import subprocess
    import sys
    script = tmp_path / "reset.py"
    script.write_text(_RESET_SCRIPT)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, str(script), root], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
