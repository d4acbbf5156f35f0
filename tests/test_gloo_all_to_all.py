"""P7: the oracle agrees with a real all-to-all collective run by CPU ranks.

Each of N processes holds one seq-sharded rank shard.  Ranks form contiguous
groups of K (review "BASP: Communication-Efficient Batch-Aware Sequence
Parallelism for LLM Training", evolve.pub, "Summary": "contiguous rank
assignment", one independent K-way all-to-all per group).  Every rank cuts its
shard into K head blocks, runs ``all_to_all_single`` on its group's process
group (gloo), and stacks the K received token blocks; the result must equal the
oracle's head-sharded shard for that rank, and the mirror exchange must bring
the seq-sharded shard back.  Ulysses is the K = N case on one N-rank group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, shape, result_dir, order="bshd"):
    B, S, H, d, N, K = shape
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        G, Bg = N // K, B // (N // K)
        Sk, Hk = S // K, H // K
        P = Bg * Sk * H * d
        groups = [dist.new_group(list(range(g * K, (g + 1) * K))) for g in range(G)]
        pg = groups[rank // K]

        x_all = synth_inputs.normal(B * S * H * d, seed=21, dtype="fp32")
        if order == "bshd":
            x = x_all[rank * P:(rank + 1) * P].view(Bg, Sk, H, d)
        else:
            # sequence-first shard [S/K, Bg, H, d], viewed batch-major for the
            # same exchange code, then stored back sequence-first
            x = x_all[rank * P:(rank + 1) * P].view(Sk, Bg, H, d).permute(1, 0, 2, 3)

        # seq -> head: send head block j' to member j'; receive token block j
        send = torch.cat([x[:, :, jp * Hk:(jp + 1) * Hk, :].reshape(-1)
                          for jp in range(K)])
        recv = torch.empty_like(send)
        dist.all_to_all_single(recv, send, group=pg)
        y5 = recv.view(K, Bg, Sk, Hk, d)          # [j][bl][sl][hl][e]
        if order == "bshd":
            y = y5.permute(1, 0, 2, 3, 4).reshape(-1)
        else:
            y = y5.permute(0, 2, 1, 3, 4).reshape(-1)  # [j][sl][bl]: s-major

        # head -> seq: send token block j to member j; receive head block j'
        if order == "bshd":
            yv = y.view(Bg, K, Sk, Hk, d)
            send2 = torch.cat([yv[:, j].reshape(-1) for j in range(K)])
        else:
            yv = y.view(K, Sk, Bg, Hk, d)
            send2 = torch.cat([yv[j].permute(1, 0, 2, 3).reshape(-1) for j in range(K)])
        recv2 = torch.empty_like(send2)
        dist.all_to_all_single(recv2, send2, group=pg)
        z5 = recv2.view(K, Bg, Sk, Hk, d)         # [j'][bl][sl][hl][e]
        if order == "bshd":
            z = z5.permute(1, 2, 0, 3, 4).reshape(-1)
        else:
            z = z5.permute(2, 1, 0, 3, 4).reshape(-1)  # [sl][bl][j'][hl][e]
        x = x_all[rank * P:(rank + 1) * P]

        ref = oracle.seq2head(synth_inputs.bits(x_all), B, S, H, d, N, K, order=order)
        ok_y = np.array_equal(synth_inputs.bits(y), ref[rank * P:(rank + 1) * P])
        ok_z = np.array_equal(synth_inputs.bits(z), synth_inputs.bits(x.reshape(-1)))
        with open(os.path.join(result_dir, "r%d" % rank), "w") as f:
            f.write("%d %d" % (ok_y, ok_z))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shape", [
    # (B, S, H, d, N, K)
    (2, 8, 4, 4, 2, 1),     # N=2, B=2: BASP K=1 (local only)
    (2, 8, 4, 4, 2, 2),     # N=2: Ulysses
    (2, 16, 8, 4, 4, 2),    # N=4, B=2: BASP, two groups of two
    (2, 16, 8, 4, 4, 4),    # N=4: Ulysses, one group of four
    (4, 8, 4, 2, 4, 2),     # N=4, B=4, two groups holding two sequences each
])
@pytest.mark.parametrize("order", ["bshd", "sbhd"])
def test_gloo_all_to_all_matches_oracle(shape, order, tmp_path):
    """The sequence-first case holds each rank's tokens as [S/K, Bg, H, d]
    (Megatron-style activations) and must match the oracle's sequence-first
    shards."""
    oracle.build()
    N = shape[4]
    mp.spawn(_worker, args=(N, _free_port(), shape, str(tmp_path), order), nprocs=N,
             join=True)
    for r in range(N):
        with open(tmp_path / ("r%d" % r)) as f:
            ok_y, ok_z = f.read().split()
        assert ok_y == "1", "rank %d: all-to-all result differs from oracle" % r
        assert ok_z == "1", "rank %d: inverse all-to-all did not restore input" % r


def _dropout_worker(rank, world, port, result_dir):
    """Rank 1 leaves before the exchange; rank 0 must see an error from its
    all-to-all within the process group's timeout instead of hanging."""
    import datetime
    import time
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    if rank == 1:
        os._exit(0)                      # dies between steps, nothing in flight
    t0 = time.time()
    outcome = "completed"
    try:
        x = torch.zeros(8)
        y = torch.empty_like(x)
        dist.all_to_all_single(y, x)
    except Exception as e:               # gloo reports the lost peer
        outcome = "error:" + type(e).__name__
    with open(os.path.join(result_dir, "r0"), "w") as f:
        f.write("%s %.1f" % (outcome, time.time() - t0))
    os._exit(0)


def test_lost_rank_is_reported_not_hung(tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_dropout_worker, args=(r, 2, port, str(tmp_path)))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank hung after its peer left")
    outcome, secs = open(tmp_path / "r0").read().split()
    assert outcome.startswith("error:"), outcome
    assert float(secs) < 60
