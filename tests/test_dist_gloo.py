"""The N > 1 path on CPU: two gloo ranks, each owning one shard of a layout.
Each rank forms its partial (sum g^2, found_inf) with the oracle (pass 1
itself needs a GPU), packs it into a zero_state_t (the library's own
host-side state init), sums it with the other rank through the package's
exchange (a real all-reduce, gloo), and steps its shard with the summed
values: with the oracle's decision and update, or with the library's own
(its host decision and element update, the code of its host-core offload
path, on a state that persists across the steps as on the device).  The
concatenated shards must equal the unpartitioned oracle step; an overflow on
one rank must skip the step on both; a rank that dies before the exchange
must make the other rank's exchange fail with an error, not hang."""
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


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, mode, out_dir, stepper="oracle"):
    import sys
    sys.path.insert(0, ROOT)
    try:
        import oracle
        import zero_partitioned_mixed_layout_gb300 as zp
        from zero_partitioned_mixed_layout_gb300.dist import exchange_partials
        import zero_synth as zs

        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                world_size=world, timeout=datetime.timedelta(seconds=10))
        numel = zs.numels(zs.tiny_transformer_shapes(hidden=64, vocab=128))
        lay = oracle.partition_layout(numel, world, 128)
        S, total = lay.shard_numel, sum(numel)
        p0 = np.zeros(lay.padded_total, np.float32)
        p0[:total] = zs.host_master(total, 0)
        p = p0[rank * S:(rank + 1) * S].copy()
        m, v = np.zeros(S, np.float32), np.zeros(S, np.float32)
        plp = np.zeros(S, np.uint16)
        hp = oracle.HParams(max_norm=0.05 if mode == "clip" else 0.0)
        zhp = zp.HParams(max_norm=hp.max_norm)
        sc = oracle.Scaler(loss_scale=1024.0)
        # the library's state, kept across the steps (library stepper)
        lstate = torch.frombuffer(bytearray(zp.zero_state_init(sc.loss_scale)), dtype=torch.uint8).clone()
        skips = []
        for k in range(3):
            # the gradient arrives multiplied by the loss scale in force:
            # the one the stepper's own state holds
            scale_now = zp.parse_state(lstate)["loss_scale"] if stepper == "library" else sc.loss_scale
            g = np.zeros(lay.padded_total, np.float16)
            g[:total] = zs.host_grad(total, 0, k, scale_now, "f16")
            if mode == "overflow" and k == 1:
                g[lay.padded_total - S + 5] = np.inf  # lands in the last rank's shard
            gr = np.ascontiguousarray(g[rank * S:(rank + 1) * S])
            if stepper == "library":
                # the partial of this rank's shard, unscaled as pass 1 leaves
                # it in the state
                sumsq, bad = oracle.norm_overflow([gr], "f16", scale_now)
                state = lstate
            else:
                sumsq, bad = oracle.norm_overflow([gr], "f16", sc.loss_scale)
                state = torch.frombuffer(bytearray(zp.zero_state_init(sc.loss_scale)),
                                         dtype=torch.uint8).clone()
            state[:16].view(torch.float64).copy_(torch.tensor([sumsq, float(bad)],
                                                              dtype=torch.float64))
            if mode == "die" and rank == 1:
                os._exit(3)  # leaves between steps, before the exchange
            exchange_partials(state)
            if stepper == "library":
                scalars = zp.zero_offload_decide(state, zhp)
                skips.append(bool(zp.parse_state(state)["last_skipped"]))
                zp.zero_offload_apply(gr, p, m, v, plp, scalars, gdtype="f16", pdtype="f16", n_threads=2)
            else:
                head = zp.parse_state(state)
                st = oracle.decide(hp, sc, head["sumsq"], int(head["found_inf"] > 0))
                skips.append(st.skip)
                oracle.adam_apply(gr, "f16", p, m, v, plp, "f16", st)
        if stepper == "library":
            final = zp.parse_state(lstate)
            step, scale = final["step"], final["loss_scale"]
        else:
            step, scale = sc.step, sc.loss_scale
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), p=p, m=m, v=v, plp=plp,
                 skips=np.array(skips), step=step, scale=scale)
        dist.destroy_process_group()
    except Exception:
        with open(os.path.join(out_dir, f"rank{rank}.err"), "w") as f:
            f.write(traceback.format_exc())
        raise


def run(mode, tmp_path, world=2, stepper="oracle"):
    port = free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=rank_main, args=(r, world, port, mode, str(tmp_path), stepper))
             for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
        if pr.is_alive():
            pr.kill()
            raise AssertionError("a rank hung")
    return [pr.exitcode for pr in procs]


def reference(mode, world=2):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import zero_synth as zs
    numel = zs.numels(zs.tiny_transformer_shapes(hidden=64, vocab=128))
    lay = oracle.partition_layout(numel, world, 128)
    total = sum(numel)
    N = lay.padded_total
    p = np.zeros(N, np.float32)
    p[:total] = zs.host_master(total, 0)
    m, v, plp = np.zeros(N, np.float32), np.zeros(N, np.float32), np.zeros(N, np.uint16)
    hp = oracle.HParams(max_norm=0.05 if mode == "clip" else 0.0)
    sc = oracle.Scaler(loss_scale=1024.0)
    for k in range(3):
        g = np.zeros(N, np.float16)
        g[:total] = zs.host_grad(total, 0, k, sc.loss_scale, "f16")
        if mode == "overflow" and k == 1:
            g[N - lay.shard_numel + 5] = np.inf
        oracle.adam_step([g], "f16", [p], [m], [v], [plp], "f16", hp, sc)
    return p, m, v, plp, sc


@pytest.mark.parametrize("stepper", ["oracle", "library"])
@pytest.mark.parametrize("mode", ["plain", "clip", "overflow"])
def test_two_gloo_ranks_equal_unpartitioned(mode, stepper, tmp_path):
    codes = run(mode, tmp_path, stepper=stepper)
    errs = [open(os.path.join(tmp_path, f)).read() for f in os.listdir(tmp_path)
            if f.endswith(".err")]
    assert codes == [0, 0], errs
    parts = [np.load(os.path.join(tmp_path, f"rank{r}.npz")) for r in range(2)]
    p, m, v, plp, sc = reference(mode)
    for key, ref in (("p", p), ("m", m), ("v", v), ("plp", plp)):
        cat = np.concatenate([q[key] for q in parts])
        if mode == "clip":
            # the two-rank norm sums two binary64 partials: within 1e-15 of
            # the sequential sum; the update within the parity tolerance
            assert np.all(np.abs(cat.astype(np.float64) - ref) <= 1e-6 * np.abs(ref) + 1e-12)
        else:
            assert cat.tobytes() == ref.tobytes(), key
    for q in parts:
        assert int(q["step"]) == sc.step and float(q["scale"]) == sc.loss_scale
    if mode == "overflow":
        # the inf sits in rank 1's shard only, yet both ranks skip step 2
        assert [list(q["skips"]) for q in parts] == [[False, True, False]] * 2


def test_dead_rank_fails_the_exchange(tmp_path):
    codes = run("die", tmp_path)
    assert codes[1] == 3
    assert codes[0] != 0, "the surviving rank should fail, not complete"
    err = open(os.path.join(tmp_path, "rank0.err")).read()
    assert "exchange_partials" in err or "all_reduce" in err
