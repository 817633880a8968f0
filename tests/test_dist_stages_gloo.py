"""ZeRO stage 2 and stage 3 exchanges across ranks, on CPU: Nd gloo ranks
move gradients and parameter shards through the package's exchanges (a
real all-to-all and all-gather, gloo) and take the arithmetic with the
oracle on each rank; the results equal the oracle on all ranks' data at
once, bit for bit."""
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


def model(world):
    import oracle
    import zero_synth as zs
    numel = zs.numels(zs.tiny_transformer_shapes(hidden=64, vocab=128))
    lay = oracle.partition_layout(numel, world, 128)
    N = lay.padded_total
    total = sum(numel)
    grads = []
    for r in range(world):
        g = np.zeros(N, np.float16)
        g[:total] = zs.host_grad(total, 40 + r, 0, 1024.0, "f16")
        grads.append(g)
    flat = np.zeros(N, np.float16)
    flat[:total] = zs.host_master(total, 41).astype(np.float16)
    return numel, lay, grads, flat


def rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    try:
        import oracle
        from zero_partitioned_mixed_layout_gb300.dist import stage2_exchange_grads, stage3_gather_shards
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                                world_size=world, timeout=datetime.timedelta(seconds=20))
        numel, lay, grads, flat = model(world)
        S = lay.shard_numel
        # stage 2: every replica of this rank's shard, then their mean
        reps = stage2_exchange_grads(torch.from_numpy(grads[rank].copy()))
        assert tuple(reps.shape) == (world, S)
        mean = oracle.reduce_mean([row.numpy() for row in reps], "f16", "f16")
        # stage 3: every rank's parameter shard, then the tensors
        shards = stage3_gather_shards(torch.from_numpy(flat[rank * S:(rank + 1) * S].copy()))
        tensors = oracle.gather_params([row.numpy() for row in shards], lay.tensor_offset, numel)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), mean=mean,
                 tensors=np.concatenate([t.view(np.uint16) for t in tensors]))
        dist.destroy_process_group()
    except Exception:
        with open(os.path.join(out_dir, f"rank{rank}.err"), "w") as f:
            f.write(traceback.format_exc())
        raise


@pytest.mark.parametrize("world", [2, 3])
def test_stage2_and_stage3_exchanges(world, tmp_path):
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
    numel, lay, grads, flat = model(world)
    S = lay.shard_numel
    whole_mean = oracle.reduce_mean(grads, "f16", "f16")
    want_tensors = np.concatenate([flat[o:o + n].view(np.uint16) for o, n in zip(lay.tensor_offset, numel)])
    for r in range(world):
        got = np.load(os.path.join(tmp_path, f"rank{r}.npz"))
        assert got["mean"].tobytes() == whole_mean[r * S:(r + 1) * S].tobytes(), f"rank {r}: stage-2 mean"
        assert got["tensors"].tobytes() == want_tensors.tobytes(), f"rank {r}: stage-3 tensors"


def test_exchanges_refuse_bad_arguments():
    """Argument checks come before any collective (no process group here)."""
    import sys
    sys.path.insert(0, ROOT)
    from zero_partitioned_mixed_layout_gb300 import dist as zdist
    with pytest.raises(ValueError):
        zdist.stage2_exchange_grads(torch.zeros(4, 8, dtype=torch.float16))
    with pytest.raises(ValueError):
        zdist.stage3_gather_shards(torch.zeros(2, 2))
    with pytest.raises(ValueError):
        zdist.onebit_exchange_worker_signs(torch.zeros(64), torch.zeros(1))
    with pytest.raises(ValueError):
        zdist.onebit_exchange_server_signs(torch.zeros(8, dtype=torch.int64), torch.zeros(1))
    with pytest.raises(ValueError):
        zdist.exchange_partials(torch.zeros(8, dtype=torch.uint8))
