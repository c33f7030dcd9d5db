"""Token-sharded data parallelism on CPU ranks (gloo, world_size 2).

The loss is a mean over counted tokens, so it shards over tokens: rank r holds
tokens T_r and computes its own sums. The global loss is
sum_r (N_r * loss_r) / sum_r N_r. Calling the backward with
grad_loss = N_r / N rescales rank r's 1/N_r normalisation to the global 1/N.
dH rows are then final, and dW is the sum over ranks (one all-reduce, the
ordinary data-parallel gradient reduction). Here every rank runs the fp64
oracle on its shard, and the reduced results must equal the whole-batch
oracle. The same host arithmetic drives the CUDA path on N GPUs (no
collective inside the library).

The two loss variants (the mixed soft + hard-label loss and the reverse KL over
the cached ids) average over the same counted tokens and are checked the same
way. Also covers bench.py's multi-rank timing rule: the reported time is the
max over ranks.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    rng = np.random.default_rng(0)
    T, d, V, K, tau = 37, 12, 50, 5, 1.5
    H = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) / np.sqrt(d)
    idx = np.stack([rng.permutation(V)[:K] for _ in range(T)])
    logit = rng.standard_normal((T, K)) * 2
    mask = (rng.random(T) < 0.7).astype(np.uint8)
    return H, W, idx, logit, mask, tau


def _labels(T, V):
    return np.random.default_rng(1).integers(0, V, size=T)


def _shard(T, rank, world):
    lo = (T * rank) // world
    hi = (T * (rank + 1)) // world
    return lo, hi


def _worker(rank, port, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import oracle.kl_oracle as ok
        H, W, idx, logit, mask, tau = _problem()
        lo, hi = _shard(H.shape[0], rank, WORLD)
        loss_r, _, kl_r = ok.forward(H[lo:hi], W, idx[lo:hi], logit[lo:hi], mask[lo:hi], tau)
        n_r = int(mask[lo:hi].sum())
        sums = torch.tensor([loss_r * n_r, float(n_r)], dtype=torch.float64)
        dist.all_reduce(sums)
        N = sums[1].item()
        loss = sums[0].item() / N
        dH_r, dW_r = ok.backward(H[lo:hi], W, idx[lo:hi], logit[lo:hi], mask[lo:hi], tau,
                                 grad_loss=n_r / N)
        dW = torch.from_numpy(dW_r)
        dist.all_reduce(dW)
        # the loss variants average over the same counted tokens, so they
        # shard the same way: the mixed loss, and the reverse KL
        labels = _labels(H.shape[0], W.shape[0])
        var = {}
        for name, fwd, bwd in (
                ("mixed",
                 lambda *a: ok.forward_mixed(*a, tau, 0.3, True, labels[lo:hi])[0],
                 lambda *a, g: ok.backward_mixed(*a, tau, 0.3, True, labels[lo:hi], g)),
                ("rkl",
                 lambda *a: ok.reverse_kl_forward(*a, tau)[0],
                 lambda *a, g: ok.reverse_kl_backward(*a, tau, g))):
            shard = (H[lo:hi], W, idx[lo:hi], logit[lo:hi], mask[lo:hi])
            s_r = torch.tensor([fwd(*shard) * n_r], dtype=torch.float64)
            dist.all_reduce(s_r)
            vdH, vdW = bwd(*shard, g=n_r / N)
            vdW = torch.from_numpy(vdW)
            dist.all_reduce(vdW)
            var[name] = (s_r.item() / N, vdH, vdW.numpy())
        # bench.py's rule: report the slowest rank's time
        t = torch.tensor([10.0 + rank], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        out_q.put((rank, loss, lo, hi, dH_r, dW.numpy(), t.item(), var))
    finally:
        dist.destroy_process_group()


def test_token_sharded_dp_matches_whole_batch():
    import oracle.kl_oracle as ok
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    H, W, idx, logit, mask, tau = _problem()
    loss, _, _ = ok.forward(H, W, idx, logit, mask, tau)
    dH, dW = ok.backward(H, W, idx, logit, mask, tau)
    labels = _labels(H.shape[0], W.shape[0])
    whole = {
        "mixed": (ok.forward_mixed(H, W, idx, logit, mask, tau, 0.3, True, labels)[0],
                  *ok.backward_mixed(H, W, idx, logit, mask, tau, 0.3, True, labels)),
        "rkl": (ok.reverse_kl_forward(H, W, idx, logit, mask, tau)[0],
                *ok.reverse_kl_backward(H, W, idx, logit, mask, tau)),
    }
    for rank, loss_g, lo, hi, dH_r, dW_g, tmax, var in res:
        assert abs(loss_g - loss) < 1e-12
        np.testing.assert_allclose(dH_r, dH[lo:hi], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dW_g, dW, rtol=1e-12, atol=1e-15)
        assert tmax == 10.0 + WORLD - 1
        for name, (l_w, dH_w, dW_w) in whole.items():
            l_g, vdH, vdW = var[name]
            assert abs(l_g - l_w) < 1e-12 * max(1.0, abs(l_w)), name
            np.testing.assert_allclose(vdH, dH_w[lo:hi], rtol=1e-11, atol=1e-14, err_msg=name)
            np.testing.assert_allclose(vdW, dW_w, rtol=1e-11, atol=1e-14, err_msg=name)


def test_rank_that_never_joins_is_reported():
    """A rank that never joins: the others' rendezvous times out with an error
    on the host (no device involved)."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_lonely, args=(_free_port(), q))
    p.start()
    msg = q.get(timeout=120)
    p.join(timeout=60)
    assert msg.startswith("error:"), msg


def _lonely(port, q):
    import datetime
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    try:
        dist.init_process_group("gloo", rank=0, world_size=2,
                                timeout=datetime.timedelta(seconds=3))
        q.put("joined")
    except Exception as e:  # noqa: BLE001 - any rendezvous failure is the expected outcome
        q.put("error: %s" % type(e).__name__)
