"""Expert parallelism across processes on CPU (gloo): the exchange the
single-GPU simulation performs in one launch, here with real collectives
between ranks.  Each rank owns the tokens [floor(r*T/R), floor((r+1)*T/R))
and the experts [r*E/R, (r+1)*E/R).  It routes its own tokens (oracle),
all-gathers the per-expert counts, sends every routed row to the rank of its
expert (all-to-all), lays the received rows out by (expert, source rank),
computes its experts' products (oracle, fp64), sends every result back, and
combines its own tokens.  The receive layout must be the oracle's exchange
layout, and every product and combined row must equal the single-process
oracle bit for bit (same fp64 arithmetic per row, same slot order)."""
import os
import socket
import traceback

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from moe_token_dispatch_persistent_gb300 import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _inputs(T, H, F, E, seed):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32))
    logits = rng.standard_normal((T, E), dtype=np.float32)
    return x, logits, W


def _a2a(send, send_counts, recv_counts, width):
    """all_to_all of rows (int64 or float64, `width` values per row)."""
    out = torch.empty((sum(recv_counts), width), dtype=send.dtype)
    dist.all_to_all_single(out, send.contiguous(), output_split_sizes=list(recv_counts),
                           input_split_sizes=list(send_counts))
    return out


def _ep_worker(rank, R, port, q, T, H, F, E, k, seed):
    try:
        _ep_rank(rank, R, port, q, T, H, F, E, k, seed)
    except Exception:  # report instead of leaving the parent waiting on the queue
        q.put((rank, "error", traceback.format_exc()))
        raise


def _ep_rank(rank, R, port, q, T, H, F, E, k, seed):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=R)
    try:
        from oracle.oracle import Oracle

        orc = Oracle()
        x, logits, W = _inputs(T, H, F, E, seed)  # every rank reads only its own slices below
        t0, t1 = T * rank // R, T * (rank + 1) // R
        epr = E // R
        # 1. route own tokens; per-expert counts of own entries
        idx, gate = orc.route(logits[t0:t1], k)
        cnt = torch.from_numpy(np.bincount(idx.ravel(), minlength=E).astype(np.int64))
        # 2. all-gather of the counts
        table = [torch.empty(E, dtype=torch.int64) for _ in range(R)]
        dist.all_gather(table, cnt)
        table = torch.stack(table).numpy()  # [R, E]
        # 3. send own entries, in (expert, t, j) order, to the rank of their expert
        order = sorted(((int(idx[i, j]), t0 + i, j) for i in range(t1 - t0) for j in range(k)))
        gid = np.array([t * k + j for _, t, j in order], dtype=np.int64)
        rows = np.stack([x[t].astype(np.int64) for _, t, _ in order]) if order else np.zeros((0, H), np.int64)
        send_counts = [int(cnt[q_ * epr:(q_ + 1) * epr].sum()) for q_ in range(R)]
        recv_counts = [int(table[s, rank * epr:(rank + 1) * epr].sum()) for s in range(R)]
        payload = np.concatenate([gid[:, None], rows], axis=1)
        got = _a2a(torch.from_numpy(payload), send_counts, recv_counts, H + 1).numpy()
        # 4. lay the received rows out by (expert, source rank): each source's
        # rows arrive in expert order, so cut them per expert and interleave
        blocks, pos = {}, 0
        for s in range(R):
            for e in range(rank * epr, (rank + 1) * epr):
                n = int(table[s, e])
                blocks[(e, s)] = got[pos:pos + n]
                pos += n
        recv = np.concatenate([blocks[(e, s)] for e in range(rank * epr, (rank + 1) * epr) for s in range(R)]
                              + [np.zeros((0, H + 1), np.int64)])
        recv_ids = recv[:, 0].copy()
        # 5. products of the rank's experts on the received rows (local problem: k = 1)
        local_counts = [int(table[:, e].sum()) for e in range(rank * epr, (rank + 1) * epr)]
        offs = np.concatenate([[0], np.cumsum(local_counts)]).astype(np.int32)
        x_recv = recv[:, 1:].astype(np.uint16)
        y = orc.expert_rows(x_recv if len(x_recv) else np.zeros((1, H), np.uint16), W[rank * epr:(rank + 1) * epr],
                            1, offs, np.arange(len(recv), dtype=np.int32), np.arange(len(recv)))
        # 6. results back to the sending ranks (each source's rows, in the order it sent them)
        back_send_counts = recv_counts
        back_recv_counts = send_counts
        per_src = {s: [] for s in range(R)}
        for e in range(rank * epr, (rank + 1) * epr):
            for s in range(R):
                n = int(table[s, e])
                start = int(offs[e - rank * epr]) + int(table[:s, e].sum())
                per_src[s].append(np.concatenate([recv_ids[start:start + n, None].astype(np.float64),
                                                  y[start:start + n]], axis=1))
        back = np.concatenate([np.concatenate(per_src[s] + [np.zeros((0, F + 1))]) for s in range(R)])
        ret = _a2a(torch.from_numpy(back), back_send_counts, back_recv_counts, F + 1).numpy()
        # 7. combine own tokens: returned rows come in the sent order, i.e. (expert, t, j)
        ret_ids = ret[:, 0].astype(np.int64)
        assert np.array_equal(ret_ids, gid)  # every entry came back, in order
        local_src = (ret_ids - t0 * k).astype(np.int32)
        local_gate = np.array([gate[t - t0, j] for _, t, j in order], dtype=np.float32)
        out = orc.combine(ret[:, 1:], local_src, local_gate, t1 - t0, k)
        q.put((rank, recv_ids, ret_ids, ret[:, 1:], out))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("R,T,E,k", [(2, 40, 8, 2), (4, 37, 8, 3), (2, 9, 4, 4)], ids=["R2", "R4_ragged", "R2_k_eq_E"])
def test_expert_parallel_exchange_matches_single_process(R, T, E, k):
    H, F, seed = 16, 8, 29
    from oracle.oracle import Oracle

    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ep_worker, args=(r, R, port, q, T, H, F, E, k, seed)) for r in range(R)]
    for p in procs:
        p.start()
    results = []
    for _ in range(R):
        r = q.get(timeout=120)
        if len(r) == 3 and r[1] == "error":
            # the other ranks may be blocked in a collective with the failed one
            for p in procs:
                p.join(timeout=5)
                if p.is_alive():
                    p.kill()
            pytest.fail(f"rank {r[0]} failed:\n{r[2]}")
        results.append(r)
    results.sort(key=lambda r: r[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0

    orc = Oracle()
    x, logits, W = _inputs(T, H, F, E, seed)
    full = orc.full(x, logits, W, k)
    _, roff, rsrc = orc.ep_layout(full["topk_idx"], E, R)
    y_of = dict(zip(full["src_index"].tolist(), full["y"]))
    ref_out = orc.combine(full["y"], full["src_index"], full["gate_w"], T, k)
    for rank, recv_ids, ret_ids, y_back, out in results:
        np.testing.assert_array_equal(recv_ids, rsrc[roff[rank]:roff[rank + 1]])
        for gid, row in zip(ret_ids.tolist(), y_back):
            np.testing.assert_array_equal(row, y_of[gid])
        np.testing.assert_array_equal(out, ref_out[T * rank // R:T * (rank + 1) // R])
