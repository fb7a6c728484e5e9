"""Multi-rank host logic on CPU: world size 2 over the gloo backend (127.0.0.1). The data path has no
collective; what the ranks exchange is the step time (max over ranks) and, offline, the per-head calibration
energy before the int8-head ranking, which must give every rank the same heads."""
import os
import socket

import numpy as np
import pytest

from pace_testlib import ensure_built

torch = pytest.importorskip("torch")

H, B_GLOBAL, DP = 32, 13, 8


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _energies():
    rng = np.random.default_rng(7)
    e = rng.lognormal(0.0, 1.0, size=(B_GLOBAL, H))      # per-sequence, per-head ||Q(S) - S||^2
    a = rng.uniform(0.85, 0.999, size=H)                  # per-head mean decay
    return e, a


def _rank_main(rank, world, port, outdir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from bit_gated_delta_gb300 import shard
    e, a = _energies()
    b0, nb = shard.batch_slice(B_GLOBAL, world, rank)
    mask = shard.assign_heads_global(e[b0:b0 + nb].sum(axis=0), nb, a, DP, 0.25, dist)
    emean = shard.global_head_energy(e[b0:b0 + nb].sum(axis=0), nb, dist)
    tmax = shard.max_over_ranks(10.0 + rank, dist)
    np.savez(os.path.join(outdir, f"r{rank}.npz"), mask=mask, emean=emean, tmax=tmax, b0=b0, nb=nb)
    dist.barrier()
    dist.destroy_process_group()


def test_batch_slice_partitions():
    from bit_gated_delta_gb300 import shard
    for B in (0, 1, 7, 64, 128, 129):
        for world in (1, 2, 3, 8):
            parts = [shard.batch_slice(B, world, r) for r in range(world)]
            assert sum(n for _, n in parts) == B
            assert all(parts[r][0] + parts[r][1] == parts[r + 1][0] for r in range(world - 1))
            assert max(n for _, n in parts) - min(n for _, n in parts) <= 1
    with pytest.raises(ValueError):
        shard.batch_slice(8, 2, 2)


def test_two_ranks_agree_on_heads_and_step_time(tmp_path):
    ensure_built()
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [np.load(os.path.join(tmp_path, f"r{r}.npz")) for r in range(world)]
    e, a = _energies()
    import bit_gated_delta_gb300 as P
    single = P.pace_assign_heads(e.mean(axis=0).astype(np.float32), a.astype(np.float32), DP, 0.25)
    for r in res:
        np.testing.assert_allclose(r["emean"], e.mean(axis=0), rtol=1e-12)
        assert np.array_equal(r["mask"], single)       # same heads on every rank as on one process
        assert float(r["tmax"]) == 11.0                # the slowest rank sets the step time
    assert int(res[0]["nb"]) + int(res[1]["nb"]) == B_GLOBAL
    assert int(single.sum()) == H // 4
