"""Seeded synthetic inputs for the fused chunked KL distillation loss.

This module draws random numbers and lays them out in the byte layout the
library consumes. It holds none of the loss's arithmetic: no softmax, no
logsumexp, no KL, no gradient. Both the CUDA path and the CPU oracle are fed
the tensors it returns, so a parity test compares the two on identical bytes.

Workloads stand in for the pages' own runs: the 8K-context Llama-3.2-3B-like
student ("Efficient knowledge distillation for LLMs: offline top-K logits and
a fused chunked KL loss", table of section "Performance and memory
benchmarks"), the GPT-OSS-20B run at 32,768 tokens and the toy
output-projection benchmark that runs to 256K tokens ("Making knowledge
distillation cheap enough to run at scale", section "Scaling to long
contexts"). The real models, teacher caches and
training data are not used: every tensor is synthetic.

Recipe (all from ``numpy.random.SeedSequence(seed)``, one child stream per
tensor, so changing one tensor's recipe leaves the others' bytes unchanged):

* H ~ N(0, 1) rounded to bf16 (round to nearest even), shape [T, d].
* W ~ N(0, 1/d) rounded to bf16, shape [V, d]; with these scales z = H.W^T
  is roughly N(0, 1).
* topk_logit: K draws of N(0, 2^2) per row, sorted in descending order (a
  teacher cache stores its top-K largest first), fp32.
* topk_idx: K distinct vocabulary ids per row, int32. ``uniform`` draws them
  uniformly. ``half_overlap`` takes floor(K/2) of them at random from the
  student's own top-K of z (computed here in fp32 only to pick ids) and the
  rest uniformly from outside that set, then shuffles the row; the first
  (largest) logit is paired with the first id after the shuffle. For K = 1 the
  single id is the student's top-1 with probability 1/2.
* mask: uint8, all ones, or for padded batches the last
  round(pad_frac * seq_len) positions of every sequence set to 0.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    V: int
    K: int
    chunk: int
    tau: float
    teacher: str  # "uniform" or "half_overlap"
    seq_len: int = 0  # >0: T is a batch of sequences of this length
    pad_frac: float = 0.0  # fraction of each sequence's tail that is masked out

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Workloads, named for what they are.
WORKLOADS = {
    # Small case the oracle finishes in well under a second.
    "small": Workload("small", T=256, d=256, V=4096, K=16, chunk=64, tau=1.0,
                      teacher="uniform"),
    # Llama-3.2-3B-like student head, 8K context, batch 1.
    "llama3b_8k": Workload("llama3b_8k", T=8192, d=3072, V=128256, K=100,
                           chunk=1024, tau=1.0, teacher="half_overlap"),
    # GPT-OSS-20B-like student head, 32K context, batch 1.
    "gptoss20b_32k": Workload("gptoss20b_32k", T=32768, d=2880, V=201088,
                              K=100, chunk=2048, tau=1.0,
                              teacher="half_overlap"),
    # Toy output projection at 256K tokens (peak memory must stay linear in T).
    "toyproj_256k": Workload("toyproj_256k", T=262144, d=4096, V=128256,
                             K=100, chunk=4096, tau=1.0, teacher="uniform"),
    # Batch of 4 x 8192 with the last 20 % of every sequence padded out.
    "padded_4x8k": Workload("padded_4x8k", T=32768, d=3072, V=128256, K=100,
                            chunk=1024, tau=1.0, teacher="half_overlap",
                            seq_len=8192, pad_frac=0.2),
}


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _distinct_rows(rng: np.random.Generator, rows: int, k: int, V: int,
                   exclude: np.ndarray | None = None) -> np.ndarray:
    """``rows`` x ``k`` ids in [0, V), distinct within a row and disjoint from
    the matching row of ``exclude`` (rows of distinct ids)."""
    n_ex = 0 if exclude is None else exclude.shape[1]
    if k + n_ex > V:
        raise ValueError("cannot draw %d distinct ids outside %d of %d" % (k, n_ex, V))
    if rows == 0 or k == 0:
        return np.zeros((rows, k), dtype=np.int64)
    if 4 * (k + n_ex) > V:
        # Dense regime: rank random keys, excluded ids pushed to the end.
        out = np.empty((rows, k), dtype=np.int64)
        for r in range(rows):
            keys = rng.random(V)
            if exclude is not None:
                keys[exclude[r]] = 2.0
            out[r] = np.argsort(keys, kind="stable")[:k]
        return out
    out = rng.integers(0, V, size=(rows, k), dtype=np.int64)
    todo = np.arange(rows)
    while True:
        cand = out[todo]
        both = cand if exclude is None else np.concatenate([cand, exclude[todo]], axis=1)
        s = np.sort(both, axis=1)
        bad = (s[:, 1:] == s[:, :-1]).any(axis=1)
        if not bad.any():
            return out
        todo = todo[bad]
        out[todo] = rng.integers(0, V, size=(len(todo), k), dtype=np.int64)


def student_topk_ids(H: torch.Tensor, W: torch.Tensor, K: int,
                     device: str | torch.device = "cpu", rows_per_block: int = 1024) -> np.ndarray:
    """Ids of the K largest entries of each row of H.W^T, in fp32 from the bf16
    values. Used only to choose which ids a synthetic teacher cache holds."""
    T = H.shape[0]
    Wd = W.to(device=device, dtype=torch.float32)
    out = np.empty((T, K), dtype=np.int64)
    for r0 in range(0, T, rows_per_block):
        h = H[r0:r0 + rows_per_block].to(device=device, dtype=torch.float32)
        out[r0:r0 + h.shape[0]] = torch.topk(h @ Wd.T, K, dim=1).indices.cpu().numpy()
    del Wd
    return out


def make_inputs(w: Workload, seed: int = 0, topk_device: str | torch.device | None = None):
    """Return a dict of CPU tensors: H [T,d] bf16, W [V,d] bf16,
    topk_idx [T,K] int32, topk_logit [T,K] fp32, mask [T] uint8."""
    T, d, V, K = w.T, w.d, w.V, w.K
    ss = np.random.SeedSequence(seed)
    r_h, r_w, r_idx, r_logit, r_pick = [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(5)]

    H = _bf16(r_h.standard_normal((T, d), dtype=np.float32))
    W = _bf16(r_w.standard_normal((V, d), dtype=np.float32) * np.float32(1.0 / math.sqrt(d)))

    logit = r_logit.standard_normal((T, K), dtype=np.float32) * np.float32(2.0)
    logit = -np.sort(-logit, axis=1)

    if w.teacher == "uniform":
        idx = _distinct_rows(r_idx, T, K, V)
    elif w.teacher == "half_overlap":
        if topk_device is None:
            topk_device = "cuda" if torch.cuda.is_available() else "cpu"
        own = student_topk_ids(H, W, K, topk_device)
        if K == 1:
            outside = _distinct_rows(r_idx, T, 1, V, exclude=own)
            coin = r_pick.random(T) < 0.5
            idx = np.where(coin[:, None], own, outside)
        else:
            n_own = K // 2
            pick = np.argsort(r_pick.random((T, K)), axis=1)[:, :n_own]
            chosen = np.take_along_axis(own, pick, axis=1)
            outside = _distinct_rows(r_idx, T, K - n_own, V, exclude=own)
            idx = np.concatenate([chosen, outside], axis=1)
            perm = np.argsort(r_pick.random((T, K)), axis=1)
            idx = np.take_along_axis(idx, perm, axis=1)
    else:
        raise ValueError("unknown teacher recipe %r" % (w.teacher,))

    mask = np.ones(T, dtype=np.uint8)
    if w.seq_len > 0 and w.pad_frac > 0:
        pad = int(round(w.pad_frac * w.seq_len))
        for s0 in range(0, T, w.seq_len):
            end = min(s0 + w.seq_len, T)
            mask[max(s0, end - pad):end] = 0

    return {
        "H": H.contiguous(),
        "W": W.contiguous(),
        "topk_idx": torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)),
        "topk_logit": torch.from_numpy(np.ascontiguousarray(logit, dtype=np.float32)),
        "mask": torch.from_numpy(mask),
    }
