"""Head-sharded (Ulysses-style) exchange of chunk_windowed_softmax_gb300.sharded on CPU, with world_size-2 gloo
process groups (no GPU): sequence shards to head shards and back, bit for bit, and the whole sharded layer with the
fp64 oracle in place of the GPU computation equals the oracle on the unsharded layer, row for row (the MiniMax-H3
Ulysses pull request, sglang #43164, Motivation: q, k, v exchanged to head shards, the output exchanged back)."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# T, S, K, r, G, global_pos: L = 7 * 5 + 3 = 38 rows, split 19 / 19 or unevenly (the exchange allows any split)
GEO = (7, 5, 2, 1, 3, 1)
B, H, D = 2, 4, 8


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def full_inputs():
    T, S, K, r, G, gp = GEO
    g = torch.Generator().manual_seed(5)
    return tuple(torch.randn(B, T * S + G, H, D, generator=g).to(torch.bfloat16) for _ in range(3))


def _worker(rank, world, port, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        import oracle.ref as ref
        from chunk_windowed_softmax_gb300 import sharded
        T, S, K, r, G, gp = GEO
        L = T * S + G
        qf, kf, vf = full_inputs()
        hn = H // world
        heads = slice(rank * hn, (rank + 1) * hn)
        for sizes in (sharded.even_seq_sizes(L, world), [11, L - 11]):
            off = sum(sizes[:rank])
            rows = slice(off, off + sizes[rank])
            x = qf[:, rows].contiguous()
            xh = sharded.seq_to_heads(x, sizes)
            assert torch.equal(xh, qf[:, :, heads]), "head shard"
            assert torch.equal(sharded.heads_to_seq(xh, sizes), x), "round trip"

            def attend(qh, kh, vh):  # the oracle on this rank's heads, whole sequence
                return torch.from_numpy(ref.window_attention(qh, kh, vh, T, S, K, r, G, gp))

            got = sharded.sharded_forward(qf[:, rows].contiguous(), kf[:, rows].contiguous(),
                                          vf[:, rows].contiguous(), T, S, K, r, G, gp, seq_sizes=sizes, attend=attend)
            want = ref.window_attention(qf, kf, vf, T, S, K, r, G, gp)[:, rows]
            assert np.array_equal(got.numpy(), want), "sharded layer"
        q.put((rank, "ok"))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent on the queue
        q.put((rank, repr(e)))


def test_sequence_head_exchange_and_sharded_layer_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: "ok", 1: "ok"}, res
    assert all(p.exitcode == 0 for p in procs)


def _worker3(rank, world, port, q):
    """Three ranks, six heads, sequence shards of unequal sizes (one of them empty): round trip."""
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from chunk_windowed_softmax_gb300 import sharded
        g = torch.Generator().manual_seed(9)
        full = torch.randn(2, 41, 6, 4, generator=g).to(torch.bfloat16)
        for sizes in (sharded.even_seq_sizes(41, world), [1, 30, 10], [20, 0, 21]):
            off = sum(sizes[:rank])
            x = full[:, off:off + sizes[rank]].contiguous()
            xh = sharded.seq_to_heads(x, sizes)
            assert torch.equal(xh, full[:, :, 2 * rank:2 * rank + 2]), "head shard"
            assert torch.equal(sharded.heads_to_seq(xh, sizes), x), "round trip"
        q.put((rank, "ok"))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:
        q.put((rank, repr(e)))


def test_exchange_three_ranks_uneven_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker3, args=(r, 3, port, q)) for r in range(3)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert res == {0: "ok", 1: "ok", 2: "ok"}, res
    assert all(p.exitcode == 0 for p in procs)


def test_even_seq_sizes():
    from chunk_windowed_softmax_gb300 import sharded
    assert sharded.even_seq_sizes(99968, 8) == [12496] * 8
    assert sharded.even_seq_sizes(38, 3) == [13, 13, 12]
    assert sum(sharded.even_seq_sizes(15077, 7)) == 15077


def test_single_rank_exchange_is_identity():
    """Without a process group (one rank) the exchanges return the tensor unchanged."""
    from chunk_windowed_softmax_gb300 import sharded
    x = full_inputs()[0]
    assert torch.equal(sharded.seq_to_heads(x, [x.shape[1]]), x)
    assert torch.equal(sharded.heads_to_seq(x, [x.shape[1]]), x)
