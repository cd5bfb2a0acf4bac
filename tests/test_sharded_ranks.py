"""The sharded-vocabulary protocol (speculative_decoding_serial_gb300/sharded.py) on gloo ranks (CPU): each
rank scores only its own rows of W for a step, the ranks merge their packed keys with an all-reduce MAX, and
every rank advances from the merged winner. The per-rank step is made from the oracle's z restricted to the
rank's rows (the CUDA kernels need a GPU); the result must be the unsharded oracle walk."""
import os
import socket
import struct

import numpy as np
import pytest
import torch.multiprocessing as mp

MARKOV, RECURRENT = 0, 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ord(f):
    u = struct.unpack("<I", struct.pack("<f", f))[0]
    if u == 0x80000000:
        u = 0
    return (~u & 0xFFFFFFFF) if (u >> 31) else (u | 0x80000000)


def _pack(key, v):
    k = (_ord(key) << 32) | (0xFFFFFFFF - v)
    return k - (1 << 64) if k >= (1 << 63) else k  # the uint64's bits as int64


def _rank_main(rank, world, port, kind, T, q, via_bench=False):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import oracle as O
    import whead_inputs as I
    from speculative_decoding_serial_gb300 import sharded as S
    V, r, B, G, seed = 333, 32, 2, 5, 17
    d = I.make_inputs(kind, V, r, B, G, seed=4)
    lo, hi = S.shard_bounds(V, world, rank)
    Ef = (d["E"].astype(np.uint32) << 16).view(np.float32)

    def step(t, s):
        # this rank's keys for step t: the oracle's z of one step from state s, noise keyed on global rows
        one = O.walk(kind, d["W"], d["E"], d["base"][:, t:t + 1].copy(), s.numpy(), A=d["A"], c=d["c"], T=T,
                     seed=seed, t0=t, want_z=True)
        keys = []
        for b in range(B):
            best = None
            for v in range(lo, hi):
                z = float(one["z"][b, 0, v])
                key = z if T == 0 else float(np.float32(np.float32(z) / np.float32(T)) + np.float32(O.gumbel(seed, b, t, v)))
                k = _pack(key, v)
                best = k if best is None or (k ^ (-(1 << 63))) > (best ^ (-(1 << 63))) else best
            keys.append(best if best is not None else -(1 << 63))  # an empty shard never wins
        return torch.tensor(keys, dtype=torch.int64)

    def advance(x, s):
        xs = x.numpy()
        if kind == MARKOV:
            return torch.from_numpy(Ef[xs].copy())
        pre = s.numpy().astype(np.float64) @ d["A"].astype(np.float64).T + Ef[xs].astype(np.float64)
        if d["c"] is not None:
            pre += d["c"].astype(np.float64)
        return torch.from_numpy(np.tanh(pre).astype(np.float32))

    walk = S.ShardedWalk(step, S.allreduce_max(), advance)
    s0 = torch.from_numpy(d["s0"].copy())
    if via_bench:
        # the benchmark's sharded leg: its rank logic times whole walks and single merges, max over ranks
        import time
        import bench

        def timer(fn):
            t = time.perf_counter()
            fn()
            return time.perf_counter() - t
        probe = torch.zeros((B,), dtype=torch.int64)
        m = bench.sharded_measure(lambda: walk.walk(s0, G)[0], lambda: S.allreduce_max()(probe), 2, 1, world,
                                  timer)
        dist.destroy_process_group()
        q.put((rank, m["tokens"].numpy(), (m["walk_s"], m["merge_s"]), (lo, hi)))
        return
    toks, states = walk.walk(s0, G)
    dist.destroy_process_group()
    q.put((rank, toks.numpy(), states.numpy(), (lo, hi)))


@pytest.mark.parametrize("world,kind,T", [(2, MARKOV, 0.0), (2, MARKOV, 1.0), (3, RECURRENT, 0.0)])
def test_sharded_walk_on_gloo_ranks_is_the_unsharded_walk(world, kind, T):
    from oracle import oracle as O
    import whead_inputs as I
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, kind, T, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, toks, states, bounds = q.get(timeout=300)
        res[rank] = (toks, states, bounds)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # the shards tile the vocabulary
    bounds = [res[r][2] for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == 333
    assert all(bounds[i][1] == bounds[i + 1][0] for i in range(world - 1))
    d = I.make_inputs(kind, 333, 32, 2, 5, seed=4)
    ref = O.walk(kind, d["W"], d["E"], d["base"], d["s0"], A=d["A"], c=d["c"], T=T, seed=17, want_state=True)
    for r in range(world):
        np.testing.assert_array_equal(res[r][0], ref["tokens"])
        np.testing.assert_allclose(res[r][1], ref["state"], rtol=0, atol=1e-6)


def test_benchmark_sharded_leg_rank_logic_on_gloo_ranks():
    """bench.py --sharded's rank logic (warm-up, barrier, timed walks and merges, max over ranks) drives the
    protocol on two gloo ranks: every rank gets the unsharded oracle's tokens and the same (slowest rank's)
    times."""
    from oracle import oracle as O
    import whead_inputs as I
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, MARKOV, 1.0, q, True)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, toks, times, bounds = q.get(timeout=300)
        res[rank] = (toks, times)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    d = I.make_inputs(MARKOV, 333, 32, 2, 5, seed=4)
    ref = O.walk(MARKOV, d["W"], d["E"], d["base"], d["s0"], T=1.0, seed=17)
    for r in range(world):
        np.testing.assert_array_equal(res[r][0], ref["tokens"])
        assert res[r][1][0] > 0 and res[r][1][1] > 0
    assert res[0][1] == res[1][1]


def test_shard_bounds_cover_the_vocabulary_on_group_boundaries():
    from speculative_decoding_serial_gb300 import sharded as S
    for V in (1, 15, 16, 17, 1000, 151936, 248064):
        for world in (1, 2, 3, 4, 8):
            bs = [S.shard_bounds(V, world, r) for r in range(world)]
            assert bs[0][0] == 0 and bs[-1][1] == V
            for (a, b), (c, _) in zip(bs, bs[1:]):
                assert b == c and (a % 16 == 0 or a == b)  # a non-empty shard starts on a group boundary
            groups = [(b - a + 15) // 16 for a, b in bs]  # the vocabulary's last group may be partial
            assert max(groups) - min(groups) <= 1


def test_key_order_survives_the_int64_transport():
    import torch
    from speculative_decoding_serial_gb300 import sharded as S
    rng = np.random.default_rng(0)
    vals = [(_ord(float(f)) << 32) | int(v) for f, v in zip(rng.standard_normal(200).astype(np.float32),
                                                            rng.integers(0, 1 << 32, 200))]
    as_i64 = torch.tensor([x - (1 << 64) if x >= (1 << 63) else x for x in vals], dtype=torch.int64)
    order = torch.argsort(S.to_ordered(as_i64)).tolist()
    assert order == sorted(range(200), key=lambda i: vals[i])
    np.testing.assert_array_equal(S.from_ordered(S.to_ordered(as_i64)).numpy(), as_i64.numpy())
