"""1-bit Adam's two sign exchanges across ranks, on CPU: Nd gloo ranks,
each a worker and the server of its chunk.  Each rank takes its worker and
server compressions with the oracle and moves the 1-bit messages through
the package's exchanges (a real all-to-all and all-gather, gloo); after two
steps every rank's parameters, momentum and errors equal the oracle's whole
step over all workers, bit for bit."""
import datetime
import os
import socket
import traceback

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
S = 2048      # chunk elements (a multiple of 32)
T_W = 50      # the last warm-up step
STEPS = 2


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def inputs(nd):
    import zero_synth as zs
    n = nd * S
    rng = np.random.default_rng(11)
    p = zs.host_master(n, 3)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = (rng.uniform(0.1, 1.0, n) * 1e-6).astype(np.float32)
    grads = [[zs.host_grad(n, 100 + r, k, 1024.0, "f16") for r in range(nd)] for k in range(STEPS)]
    return p, m, v, grads


def rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    try:
        import oracle
        from zero_partitioned_mixed_layout_gb300.dist import (exchange_partials, onebit_exchange_server_signs,
                                                              onebit_exchange_worker_signs)
        import zero_partitioned_mixed_layout_gb300 as zp
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                world_size=world, timeout=datetime.timedelta(seconds=20))
        p, m, v, grads = inputs(world)
        n = world * S
        e_w = np.zeros(n, np.float32)
        e_s = np.zeros(S, np.float32)
        hp = oracle.HParams()
        sc = oracle.Scaler(loss_scale=1024.0, step=T_W)
        plp = np.zeros(n, np.uint16)
        for k in range(STEPS):
            g = grads[k][rank]
            # the overflow flag and norm of the local gradient, summed over ranks
            sumsq, bad = oracle.norm_overflow([g], "f16", sc.loss_scale)
            state = torch.frombuffer(bytearray(zp.zero_state_init(sc.loss_scale)), dtype=torch.uint8).clone()
            state[:16].view(torch.float64).copy_(torch.tensor([sumsq, float(bad)], dtype=torch.float64))
            exchange_partials(state)
            head = zp.parse_state(state)
            st = oracle.frozen_variance(oracle.decide(hp, sc, head["sumsq"], int(head["found_inf"] > 0)), hp, T_W)
            bits, scale = oracle.onebit_worker(g, "f16", st, m, e_w)
            chunk_bits, worker_scales = onebit_exchange_worker_signs(
                torch.from_numpy(bits.view(np.int32).copy()), torch.tensor([scale], dtype=torch.float32))
            sbits, sscale = oracle.onebit_server([row.numpy().view(np.uint32) for row in chunk_bits],
                                                 list(worker_scales.numpy()), e_s)
            all_bits, server_scales = onebit_exchange_server_signs(
                torch.from_numpy(sbits.view(np.int32).copy()), torch.tensor([sscale], dtype=torch.float32))
            oracle.onebit_update(all_bits.numpy().view(np.uint32), list(server_scales.numpy()), S, n, p, m, v,
                                 plp, "f16", st)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), p=p, m=m, plp=plp, e_w=e_w, e_s=e_s)
        dist.destroy_process_group()
    except Exception:
        with open(os.path.join(out_dir, f"rank{rank}.err"), "w") as f:
            f.write(traceback.format_exc())
        raise


@pytest.mark.parametrize("world", [2, 3])
def test_onebit_exchanges_equal_the_whole_step(world, tmp_path):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    port = free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
        if pr.is_alive():
            pr.kill()
            raise AssertionError("a rank hung")
    errs = [open(os.path.join(tmp_path, f)).read() for f in os.listdir(tmp_path) if f.endswith(".err")]
    assert [pr.exitcode for pr in procs] == [0] * world, errs
    # the oracle's step over all workers at once
    p, m, v, grads = inputs(world)
    n = world * S
    e_w = [np.zeros(n, np.float32) for _ in range(world)]
    e_s = [np.zeros(S, np.float32) for _ in range(world)]
    plp = np.zeros(n, np.uint16)
    hp, sc = oracle.HParams(), oracle.Scaler(loss_scale=1024.0, step=T_W)
    for k in range(STEPS):
        oracle.onebit_step(grads[k], "f16", S, n, p, m, v, e_w, e_s, plp, "f16", hp, sc, T_W)
    for r in range(world):
        got = np.load(os.path.join(tmp_path, f"rank{r}.npz"))
        for key, want in (("p", p), ("m", m), ("plp", plp), ("e_w", e_w[r]), ("e_s", e_s[r])):
            assert got[key].tobytes() == want.tobytes(), f"rank {r}: {key}"
