"""Data-parallel path on CPU ranks (gloo, world size 2): the token shards of
every rank tile [0, M) in whole 128-token blocks, and the all-reduced Wgrad
partials of the shards equal the Wgrad of all tokens (computed here with the
oracle, which stands in for the GPU kernels on CPU ranks)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from fp8_precision_pretraining_amax_b300.dp import allreduce_wgrad_, token_shard


@pytest.mark.parametrize("M,world", [(128, 1), (1024, 2), (1152, 2), (32768, 8), (640, 3), (384, 4)])
def test_token_shards_tile_the_tokens(M, world):
    bounds = [token_shard(M, r, world) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == M
    for (a0, a1), (b0, b1) in zip(bounds, bounds[1:]):
        assert a1 == b0
    sizes = [m1 - m0 for m0, m1 in bounds]
    assert all(s % 128 == 0 for s in sizes)
    assert max(sizes) - min(sizes) <= 128


def test_token_shard_rejects_partial_blocks():
    with pytest.raises(ValueError):
        token_shard(200, 0, 2)
    with pytest.raises(ValueError):
        token_shard(256, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_path):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(77)                     # same full problem on every rank
        M, N, K = 640, 256, 384
        mags = rng.integers(0, 0x7F, size=(N + K, M), dtype=np.uint8)
        signs = rng.integers(0, 2, size=(N + K, M), dtype=np.uint8) << 7
        codes = mags | signs
        dyqT, xqT = codes[:N], codes[N:]
        sdyT = (rng.uniform(1, 2, (M // 128, N)) * 2.0 ** rng.integers(-8, 2, (M // 128, N))).astype(np.float32)
        sxT = (rng.uniform(1, 2, (M // 128, K)) * 2.0 ** rng.integers(-8, 2, (M // 128, K))).astype(np.float32)
        m0, m1 = token_shard(M, rank, world)
        part, _ = oracle.gemm_wgrad(np.ascontiguousarray(dyqT[:, m0:m1]), sdyT[m0 // 128:m1 // 128],
                                    np.ascontiguousarray(xqT[:, m0:m1]), sxT[m0 // 128:m1 // 128])
        dw = torch.from_numpy(np.ascontiguousarray(part))
        allreduce_wgrad_(dw)
        if rank == 0:
            full, absd = oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT)
            err = np.max(np.abs(dw.numpy() - full) / (absd + 1e-300))
            np.save(result_path, np.array([err, m1 - m0]))
    finally:
        dist.destroy_process_group()


def test_wgrad_partials_allreduce_to_the_full_wgrad(tmp_path):
    world = 2
    out = str(tmp_path / "result.npy")
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    err, first_shard = np.load(out)
    assert first_shard == 384                              # 5 blocks over 2 ranks: 3 + 2
    assert err < 1e-12                                     # binary64 sums in a different order
