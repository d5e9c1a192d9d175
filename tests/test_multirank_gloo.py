"""The multi-rank path on CPU: two `gloo` ranks in spawned processes.

* bench.max_over_ranks, the reduction the benchmark applies to every timed
  quantity when it runs as several ranks, gives each rank the slowest rank's
  values; bench.whole_job_tflops counts every rank's work.
* The one exchange that sharding attention along the keys would need: each
  rank attends to its share of the key blocks (the oracle's block-list path,
  global causal mask), the ranks all-gather (O, LSE) and merge them with the
  pages' blockwise merge (oracle.attention.merge_partials); every rank then
  holds attention over all keys.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist
    import bench
    from oracle import attention as A
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(dist, [10.0 + rank, 5.0 - rank], "cpu")
        # attention sharded over key blocks: rank r owns blocks [2r, 2r + 2) of 4
        rng = np.random.default_rng(3)
        B, H, S, D, bs = 1, 2, 16, 8, 4
        q, k, v = (rng.standard_normal((B, H, S, D)) for _ in range(3))
        idx = np.full((B, H, S // bs, 2), -1, np.int32)
        idx[..., :] = np.arange(2 * rank, 2 * rank + 2, dtype=np.int32)
        o, lse = A.attention_fwd(q, k, v, 0.4, mask=A.MASK_CAUSAL, kv_block_idx=idx, block=bs)
        lse = np.where(np.isposinf(lse), -np.inf, lse)          # a shard without keys weighs 0
        mine = torch.from_numpy(np.concatenate([o.ravel(), lse.ravel()]))
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        n_o = o.size
        o_parts = np.stack([p[:n_o].numpy().reshape(o.shape) for p in parts])
        l_parts = np.stack([p[n_o:].numpy().reshape(lse.shape) for p in parts])
        merged_o, merged_l = A.merge_partials(o_parts, l_parts)
        full_o, full_l = A.attention_fwd(q, k, v, 0.4, mask=A.MASK_CAUSAL)
        ok = bool(np.allclose(merged_o, full_o, rtol=1e-12, atol=1e-13) and
                  np.allclose(merged_l, full_l, rtol=1e-12, atol=1e-13))
        out.put((rank, slowest, ok, bench.whole_job_tflops(world, 2e9, 1.0)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, ok, tflops in results:
        assert slowest == [11.0, 5.0], (rank, slowest)   # max of (10, 11) and (5, 4)
        assert ok, rank
        assert tflops == pytest.approx(4.0)                # 2 ranks x 2 GFLOP in 1 ms
