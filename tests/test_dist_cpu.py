"""The multi-process benchmark path on CPU (gloo, world_size 2): ranks meet at
the barrier, the step time is the slowest rank's, and the whole-job value
counts every rank's tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    ms = [2.0, 3.5][rank]  # the second rank is slower
    slow = bench.max_over_ranks(ms, world, device="cpu")
    out[rank] = (slow, bench.whole_job_throughput(8192, world, slow))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_value():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.5
    assert res[0][1] == pytest.approx(8192 * 2 / 3.5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.whole_job_throughput(128, 1, 0.5) == pytest.approx(256000.0)


def _ep_layer():
    """One small seeded layer, the same on every rank: 6 experts, top-3."""
    import numpy as np
    from oracle import nvfp4_oracle as O
    from nvfp4_mixture_experts_expert_gb300 import workloads as W
    wl = W.moe_workload(40, 64, 32, 6, 3, 19)
    hidden = W.bf16_bits_to_f32(wl.hidden)
    w13q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w13))
    w2q = O.quantize_expert_weights(W.bf16_bits_to_f32(wl.w2))
    a1, a2 = O.calibrate_activation_scales(hidden, wl.logits, wl.top_k, w13q)
    ids, w = O.route(wl.logits, wl.top_k)
    return np, O, wl, hidden, w13q, w2q, a1, a2, ids, w


def _ep_worker(rank, world, port, out):
    """Rank r holds experts [3r, 3r + 3) and runs the routed forward on the
    global top-k; the partial sums meet in an all-reduce."""
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    np, O, wl, hidden, w13q, w2q, a1, a2, ids, w = _ep_layer()
    per = wl.E // world
    lo = rank * per
    loc_ids, loc_w = O.remap_global_ids(ids, w, lo, per)
    sl = slice(lo, lo + per)
    part = tuple(x[sl] for x in w13q[:2]) + (w13q[2][sl],)
    part2 = tuple(x[sl] for x in w2q[:2]) + (w2q[2][sl],)
    # each rank calibrates its own experts from the same global ids
    c1, c2 = O.calibrate_activation_scales_routed(hidden, loc_ids, part)
    scales = [torch.zeros(2 * per, dtype=torch.float32) for _ in range(world)]
    dist.all_gather(scales, torch.from_numpy(np.concatenate([c1, c2]).astype(np.float32)))
    _, inter = O.moe_forward_routed(hidden, loc_ids, loc_w, part, part2, a1[sl], a2[sl], return_intermediates=True)
    acc = torch.from_numpy(inter["acc"].copy())
    dist.all_reduce(acc)
    out[rank] = (acc.numpy().tolist(), [x.numpy().tolist() for x in scales])
    dist.barrier()
    dist.destroy_process_group()


def test_expert_parallel_partial_sums_add_up_to_the_whole_layer():
    """Two gloo ranks, each with half of the experts: the sum of their routed
    forwards' FP64 accumulators equals the single-process layer's, and the
    scales each rank calibrates for its experts are the whole layer's."""
    import numpy as np
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_ep_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    np_, O, wl, hidden, w13q, w2q, a1, a2, ids, w = _ep_layer()
    _, whole = O.moe_forward_routed(hidden, ids, w, w13q, w2q, a1, a2, return_intermediates=True)
    per = wl.E // 2
    for r in (0, 1):
        acc, scales = res[r]
        np.testing.assert_allclose(np.array(acc), whole["acc"], rtol=1e-12, atol=1e-15)
        for q in (0, 1):
            np.testing.assert_array_equal(np.float32(scales[q][:per]), a1[q * per:(q + 1) * per])
            np.testing.assert_array_equal(np.float32(scales[q][per:]), a2[q * per:(q + 1) * per])
    assert np.abs(whole["acc"]).max() > 0
