"""bench.py's multi-rank logic on CPU: two gloo ranks (replicas), the step time is the slowest
rank's and the job value sums the replicas' work over it."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, ws, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    wsz, r, local = bench._dist()
    assert (wsz, r, local) == (ws, rank, rank)
    ms = 100.0 + 25.0 * rank                      # rank 1 is the slower replica
    worst = bench.reduce_max_over_ranks(ms, ws, torch.device("cpu"))
    results[rank] = (worst, bench.job_tflops(2.341e14, worst, ws))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_aggregate():
    ws = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.spawn(_rank, args=(ws, port, results), nprocs=ws, join=True)
    assert results[0][0] == results[1][0] == 125.0
    assert results[0][1] == pytest.approx(2 * 2.341e14 / 0.125 / 1e12)


def test_single_rank_is_identity():
    assert bench.reduce_max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)


def test_kernel_choice_and_stored_traffic_follow_the_library_rule():
    # bench.py names the attention kernel a run uses with the library's default rule (CTA pairs
    # for split operands, or for fp16 operands with N >= 65536) and reports the stored DRAM
    # traffic only for the kernel variant, K rotation mode and workload it was captured on.
    import argparse
    from video_diffusion_transformer_rope_gb300 import configs
    args = argparse.Namespace(kernel="default", window=None, subset=None, k_rope="prepass")
    assert bench._kernel_used(args, configs.WAN14B_720P) == "pair"
    assert bench._kernel_used(args, configs.LONG_STRESS) == "pair"
    assert bench._kernel_used(args, configs.WAN13B_480P) == "single"
    assert bench._kernel_used(argparse.Namespace(**{**vars(args), "k_rope": "fused"}), configs.WAN13B_480P) == "pair"
    assert bench._kernel_used(argparse.Namespace(**{**vars(args), "window": "2,6,10"}), configs.WAN14B_720P) == "single"
    assert bench._kernel_used(argparse.Namespace(**{**vars(args), "kernel": "single"}), configs.WAN14B_720P) == "single"
    t = bench._traffic_per_launch("wan14b_720p", "pair")
    assert t is None or 6.2e9 <= t <= 9e9          # algorithmic bytes are 6.22 GB per launch
    assert bench._traffic_per_launch("wan14b_720p", "single") is None
    assert bench._traffic_per_launch("wan1.3b_480p", "pair") is None
    assert bench._traffic_per_launch("wan14b_720p", "pair", "fused") is None   # another K mode
