"""The benchmark's multi-rank path on CPU: gloo, world size 2, no GPU.

Each rank runs an independent problem (weak scaling); the step time is the
maximum over ranks and the work is the sum over ranks.
"""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    step_ms = 10.0 + rank            # rank 1 is the slowest
    flops = 1e12 * (rank + 1)
    bench.barrier(world)
    out[rank] = (bench.reduce_max(step_ms, world), bench.reduce_sum(flops, world))
    dist.destroy_process_group()


def test_max_time_and_total_work_over_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        assert out[r] == (11.0, 3e12)


def test_visible_key_count_matches_the_workload_figures():
    import torch
    import bench
    import msa_synth as synth
    # 32K causal sink: 4 * 128 * 16 * visible keys = 2.0664e12 effective FLOP
    spec = synth.CAUSAL_SINK_32K
    q2k = synth.make_prefill_q2k(spec)
    assert abs(bench.prefill_flops(spec, q2k) - 2.0664e12) / 2.0664e12 < 1e-3
    # tiny non-causal: every selected block fully visible
    t = synth.TINY_NONCAUSAL_1K
    q2k = synth.make_prefill_q2k(t)
    assert bench.prefill_flops(t, q2k) == 4 * 128 * 2 * 1024 * 4 * 128
    # a duplicate and an out-of-range id add nothing
    q = torch.tensor([[[[0, 0, 9, -1]]]], dtype=torch.int32)
    kv = torch.tensor([1024])
    assert int(bench.visible_keys(q, 1, kv, False).sum()) == 128


def test_decode_unique_and_gathered_bytes_on_a_hand_case():
    import torch
    import bench
    import msa_synth as synth
    # one sequence of 200 used keys (block 0: 128 tokens, block 1: 72), one KV
    # head, two queries selecting {0, 1} and {1} (with padding and a repeat)
    spec = synth.DecodeSpec("hand", B=1, Sq=2, Hkv=1, qpk=1, topk=3, kv_len=217, trim=17)
    q2k = torch.tensor([[[[0, 1, -1], [1, 1, -1]]]], dtype=torch.int32)
    su = torch.tensor([200], dtype=torch.int32)
    row = spec.D * 2 * 2  # K and V bytes of one token of one head
    assert bench.decode_gathered_bytes(spec, q2k, su) == (128 + 72 + 72) * row
    unique_kv = (128 + 72) * row
    other = 2 * 2 * spec.Hq * spec.D * 2 + 2 * spec.Hq * 4 + q2k.numel() * 4 + 2 * 4
    assert bench.decode_bytes(spec, q2k, su) == unique_kv + other
