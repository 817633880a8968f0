"""The C ABI on the CPU (no GPU calls): the library builds and loads, exports
every function that include/zero_pml.h declares, and its host-only entry
points (layout, state init, workspace size, error strings) agree with the
oracle and reject bad arguments."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import zero_synth as zs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zp():
    from zero_partitioned_mixed_layout_gb300 import _build
    _build.build()
    import zero_partitioned_mixed_layout_gb300 as zp
    zp.lib()
    return zp


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(zp):
    names = declared_functions()
    assert "zero_adam_step" in names and "zero_partition_layout" in names
    so = ctypes.CDLL(zp.LIB_PATH)
    for name in names:
        assert hasattr(so, name), f"{name} declared in include/ but not exported"


def test_library_targets_sm103a(zp):
    """The kernels are compiled for sm_103a alone (one -gencode, no PTX for
    other targets), and the build passes that to every nvcc call."""
    from zero_partitioned_mixed_layout_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    src = open(_build.__file__).read()
    assert src.count("ARCH +") + src.count("+ ARCH") >= 1


@pytest.mark.parametrize("seed", range(12))
def test_layout_matches_oracle(zp, seed):
    rng = np.random.default_rng(100 + seed)
    k = int(rng.integers(0, 60))
    numel = [int(x) for x in rng.integers(0, 5000, k)]
    nd = int(rng.integers(1, 33))
    align = int(2 ** rng.integers(0, 9))
    ours = zp.zero_partition_layout(numel, nd, align)
    ref = oracle.partition_layout(numel, nd, align)
    assert ours.shard_numel == ref.shard_numel
    assert ours.padded_total == ref.padded_total
    assert list(ours.tensor_offset) == ref.tensor_offset
    assert [tuple(int(x) for x in r) for r in ours.frags] == ref.frags


@pytest.mark.parametrize("name", ["tiny", "gpt2_1p5b_nd16", "stack_100b_nd400", "frag_10k"])
def test_workload_layouts_match_oracle(zp, name):
    w = zs.WORKLOADS[name]
    numel = w["numel"]()
    ours = zp.zero_partition_layout(numel, w["nd"], w["align"])
    ref = oracle.partition_layout(numel, w["nd"], w["align"])
    assert ours.shard_numel == ref.shard_numel and ours.padded_total == ref.padded_total
    assert [tuple(int(x) for x in r) for r in ours.frags] == ref.frags


def test_layout_errors(zp):
    lib = zp.lib()
    i64 = ctypes.c_int64
    arr = (i64 * 2)(5, 7)
    s, p, nf = i64(), i64(), i64()
    def call(numel, n, nd, align, frags=None, cap=0, outs=True):
        return lib.zero_partition_layout(numel, n, nd, align, ctypes.byref(s) if outs else None,
                                         ctypes.byref(p), None, frags, cap, ctypes.byref(nf))
    # S = ceil(12 / 32) * 8 = 8: tensor 1 straddles ranks 0 and 1 -> 3 pieces
    assert call(arr, 2, 4, 8) == -6  # capacity 0 with pieces to write
    assert nf.value == 3 and s.value == 8 and p.value == 32
    assert call(arr, 2, 0, 8) == -8
    assert call(arr, 2, 4, 3) == -8
    assert call(arr, 2, 4, 0) == -8
    assert call(None, 2, 4, 8) == -1
    assert call(arr, -1, 4, 8) == -1
    assert call(arr, 2, 4, 8, outs=False) == -1
    neg = (i64 * 2)(5, -1)
    assert call(neg, 2, 4, 8) == -1
    huge = (i64 * 2)(1 << 62, 1 << 61)  # total past 2^62
    assert call(huge, 2, 4, 8) == -8


def test_state_init(zp):
    st = zp.parse_state(zp.zero_state_init(65536.0))
    assert st["loss_scale"] == 65536.0 and st["step"] == 0 and st["sumsq"] == 0.0
    assert st["last_clip"] == 1.0
    for bad in (0.0, 0.5, 3.0, float("inf"), float("nan"), -2.0):
        with pytest.raises(zp.ZeroError):
            zp.zero_state_init(bad)


def test_workspace_bytes(zp):
    a = zp.zero_workspace_bytes(1, 1000)
    b = zp.zero_workspace_bytes(1, 1 << 30)
    c = zp.zero_workspace_bytes(10_000, 1 << 30)
    d = zp.zero_workspace_bytes(10_000, 1000)
    # the table region holds a list's table (O(tensors)) or a flat pass's
    # block partials (O(elements)), whichever is larger
    assert 0 < a < b <= c and a < d <= c
    assert d - a >= 10_000 * 48 + 2 * 10_001 * 8 - 4096
    assert b - a >= ((1 << 30) - 1000) // 256 - 512
    assert all(x % 256 == 0 for x in (a, b, c, d))


def test_error_strings(zp):
    for code in range(0, -10, -1):
        s = zp.zero_strerror(code)
        assert s and s != "unknown error code"
    assert zp.zero_strerror(-99) == "unknown error code"


def test_binding_refuses_host_tensors(zp):
    torch = pytest.importorskip("torch")
    t = torch.zeros(16)
    st, ws = torch.zeros(64, dtype=torch.uint8), torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(ValueError):
        zp.zero_grad_norm_overflow(t, st, ws)
    with pytest.raises(ValueError):
        zp.zero_accumulate_grads_norm(t, [torch.zeros(16, dtype=torch.float16)], st, ws, True)
    with pytest.raises(ValueError):
        zp.zero_step(torch.zeros(16, dtype=torch.float16), t, t.clone(), t.clone(), None, zp.HParams(), st, ws)


# ---------------------------------------------------------------- stage-3 gather plan (host only)

def _plan_as_oracle(plan, n_layers):
    out = [[] for _ in range(n_layers)]
    for L, r, so, ln, lo in plan.pieces:
        out[int(L)].append((int(r), int(so), int(ln), int(lo)))
    return out


@pytest.mark.parametrize("seed", range(12))
def test_gather_plan_matches_oracle(zp, seed):
    rng = np.random.default_rng(300 + seed)
    k = int(rng.integers(0, 40))
    numel = [int(x) for x in rng.integers(0, 3000, k)]
    nd = int(rng.integers(1, 20))
    align = int(2 ** rng.integers(0, 8))
    cuts = sorted(int(x) for x in rng.integers(0, k + 1, int(rng.integers(0, 6))))
    layer_first = [0] + cuts + [k]
    ours = zp.zero_gather_plan(numel, layer_first, nd, align)
    ref = oracle.gather_plan(numel, layer_first, nd, align)
    assert _plan_as_oracle(ours, len(ref)) == [lg.pieces for lg in ref]
    assert list(ours.layer_flat) == [lg.begin for lg in ref] + [ref[-1].end]
    assert ours.max_layer_numel == max(lg.end - lg.begin for lg in ref)


def test_gather_plan_gpt2_matches_oracle(zp):
    numel = zs.WORKLOADS["gpt2_1p5b_nd16"]["numel"]()
    lf = zs.gpt2_layer_first()
    ours = zp.zero_gather_plan(numel, lf, 16, 128)
    ref = oracle.gather_plan(numel, lf, 16, 128)
    assert _plan_as_oracle(ours, len(ref)) == [lg.pieces for lg in ref]
    assert ours.max_layer_numel == (50257 + 1024) * 1600


def test_gather_plan_errors(zp):
    lib = zp.binding._gather_lib()
    i64 = ctypes.c_int64
    numel = (i64 * 3)(5, 3, 7)
    n = i64()
    for lf in ([0, 2, 1, 3], [0, 4], [-1, 3]):
        arr = (i64 * len(lf))(*lf)
        assert lib.zero_gather_plan(numel, 3, arr, len(lf) - 1, 2, 2, None, None, 0, ctypes.byref(n),
                                    None) == -8
    arr = (i64 * 2)(0, 3)
    assert lib.zero_gather_plan(numel, 3, arr, 1, 0, 2, None, None, 0, ctypes.byref(n), None) == -8
    assert lib.zero_gather_plan(numel, 3, arr, 1, 2, 2, None, None, 0, None, None) == -1
    # too small an output array: the count still comes back
    assert lib.zero_gather_plan(numel, 3, arr, 1, 2, 2, None, None, 0, ctypes.byref(n), None) == -6
    assert n.value == 2


def test_gather_workspace_bytes(zp):
    a = zp.zero_gather_workspace_bytes(580, 16)
    assert a % 256 == 0 and a >= 580 * 32 + 16 * 8
    assert zp.zero_gather_workspace_bytes(0, 1) >= 256
    assert zp.zero_gather_workspace_bytes(10_000, 400) > zp.zero_gather_workspace_bytes(10_000, 1)


def test_plan_struct_layout_matches_the_header(zp, tmp_path):
    """The binding's copy of zero_list_plan_t has the C struct's size and
    field offsets (compiled from the header with gcc)."""
    import ctypes
    import os
    import subprocess
    from zero_partitioned_mixed_layout_gb300 import binding
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "zero_pml.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu\\n", sizeof(zero_list_plan_t), '
                   'offsetof(zero_list_plan_t, one), offsetof(zero_list_plan_t, n), '
                   'offsetof(zero_list_plan_t, gdtype)); return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    P = binding._ListPlan
    assert got == [ctypes.sizeof(P), P.one.offset, P.n.offset, P.gdtype.offset]


def _comment_before(header: str, name: str) -> str:
    """The comment block that ends right before the declaration of `name`."""
    import re
    m = re.search(r"/\*((?:(?!\*/).)*)\*/\s*(?:int|size_t|const char \*)\s*" + name + r"\(", header, re.S)
    assert m, f"no comment block right before {name}"
    return m.group(1)


@pytest.mark.parametrize("name", ["zero_partition_layout", "zero_workspace_bytes", "zero_accumulate_grads",
                                  "zero_grad_norm_overflow", "zero_adam_step", "zero_step"])
def test_hot_path_calls_cite_their_passage(name):
    """Every call of the hot path's boundary states, in its header comment,
    the passage of the pages it implements ([ZeRO card §...] or [DS news])."""
    import os
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "zero_pml.h")
    block = _comment_before(open(inc, encoding="utf-8").read(), name)
    assert "[ZeRO card §" in block or "[DS news]" in block, name
