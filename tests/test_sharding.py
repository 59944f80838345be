"""Head-sharded decode across ranks (fp8_kv_cache_reshape_gb300/sharding.py):
the partition covers every KV head and query head exactly once with whole
query-head groups, and -- run as world-size-2 gloo ranks on the CPU -- each
rank's oracle decode over its heads' caches, concatenated along the head
axis, is the unsharded oracle decode bit for bit.  ("kv-cache-quantization-
fp8-scale-granularity": the KV cache is partitioned across tensor-parallel
ranks.)"""
import importlib.util
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sharding():
    # by path: the module is host logic and does not need the built library
    spec = importlib.util.spec_from_file_location(
        "kvq_sharding", os.path.join(ROOT, "fp8_kv_cache_reshape_gb300", "sharding.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # dataclasses look their module up by name
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("hq,hkv,world", [(32, 8, 1), (32, 8, 2), (32, 8, 4), (32, 8, 8), (64, 8, 8), (4, 1, 1),
                                          (16, 4, 2)])
def test_partition_covers_every_head_once_in_whole_groups(hq, hkv, world):
    sh = _sharding().all_shards(hq, hkv, world)
    kv = [h for s in sh for h in range(s.kv0, s.kv1)]
    q = [h for s in sh for h in range(s.q0, s.q1)]
    assert kv == list(range(hkv)) and q == list(range(hq))
    g = hq // hkv
    for s in sh:
        assert s.q0 == s.kv0 * g and s.q1 == s.kv1 * g  # query head h reads KV head h // g
        assert s.kv_heads == hkv // world


@pytest.mark.parametrize("hq,hkv,world", [(32, 8, 3), (30, 8, 2), (32, 8, 16), (32, 8, 0)])
def test_impossible_partitions_are_refused(hq, hkv, world):
    with pytest.raises(ValueError):
        _sharding().kv_head_shard(hq, hkv, world, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    import workloads as W
    from oracle import kv_cache
    cfg = W.DecodeConfig("shard_case", batch=3, q_heads=16, kv_heads=4, head_dim=64, context=700, outliers=2)
    case = W.decode_case(cfg, lengths=[700, 33, 400])
    kc = np.zeros((case.num_blocks, 4, 16, 64), np.uint8)
    vc = np.zeros((case.num_blocks, 4, 64, 16), np.uint8)
    kv_cache.reshape_and_cache(case.k.float().numpy(), case.v.float().numpy(), case.slot_mapping.numpy(), kc, vc,
                               case.k_scale.numpy(), case.v_scale.numpy())
    return case, kc, vc


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    from oracle import attention
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case, kc, vc = _problem()
        s = _sharding().kv_head_shard(16, 4, world, rank)
        # this rank holds only its KV heads' pages and scales, and its query heads
        kc_r = np.ascontiguousarray(kc[:, s.kv0:s.kv1])
        vc_r = np.ascontiguousarray(vc[:, s.kv0:s.kv1])
        outs = {}
        for mode in ("mirror", "pure"):
            o, lse = attention.paged_decode(case.q.float().numpy()[:, s.q0:s.q1], kc_r, vc_r,
                                            case.k_scale.numpy()[s.kv0:s.kv1], case.v_scale.numpy()[s.kv0:s.kv1],
                                            case.block_table.numpy(), case.seq_lens.numpy(), case.sm_scale,
                                            mode=mode)
            parts = [torch.zeros(3, 8, 64, dtype=torch.float64) for _ in range(world)]
            dist.all_gather(parts, torch.from_numpy(o))  # test-side gather: the kernels need none
            outs[mode] = torch.cat(parts, dim=1).numpy()
        if rank == 0:
            ok = True
            for mode in ("mirror", "pure"):
                whole, _ = attention.paged_decode(case.q.float().numpy(), kc, vc, case.k_scale.numpy(),
                                                  case.v_scale.numpy(), case.block_table.numpy(),
                                                  case.seq_lens.numpy(), case.sm_scale, mode=mode)
                ok = ok and np.array_equal(outs[mode], whole)
            q.put(ok)
    finally:
        dist.destroy_process_group()


def test_two_ranks_concatenate_to_the_unsharded_decode_bit_for_bit():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    assert q.get(timeout=5) is True
