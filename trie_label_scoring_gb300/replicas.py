"""Replica sharding of documents across GPUs (host side).

Quail runs a full model copy per GPU and has the coordinator assign documents
by their token lengths to balance the work; results are merged on the host
(Quail docs, "Execution", section "Multiple GPUs"). trie_tree has no exchange
step between documents, so this is all the multi-GPU path needs: a balanced
partition, one classify call per rank on its own documents, and a gather of
the per-document outputs back into input order. No collective touches the
data path; torch.distributed (gloo on CPU, NCCL on GPUs) only gathers results.
"""
from __future__ import annotations

import heapq

import numpy as np


def partition_by_length(doc_len, world: int) -> list:
    """Greedy longest-first assignment: each document goes to the rank with the
    fewest tokens so far (ties: lowest rank). Returns one ascending index array
    per rank; every document appears exactly once."""
    lens = np.asarray(doc_len, dtype=np.int64)
    if world <= 0:
        raise ValueError("world must be positive")
    order = sorted(range(len(lens)), key=lambda i: (-int(lens[i]), i))
    heap = [(0, r) for r in range(world)]
    shards = [[] for _ in range(world)]
    for i in order:
        load, r = heapq.heappop(heap)
        shards[r].append(i)
        heapq.heappush(heap, (load + int(lens[i]), r))
    return [np.array(sorted(s), dtype=np.int64) for s in shards]


def shard_tokens(doc_len, shards) -> list:
    lens = np.asarray(doc_len, dtype=np.int64)
    return [int(lens[s].sum()) for s in shards]


def gather_rows(local: np.ndarray, shard: np.ndarray, num_docs: int, group=None) -> np.ndarray:
    """All-gathers per-document rows (local[k] belongs to document shard[k])
    from every rank and returns them in document order, on every rank."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    local = np.ascontiguousarray(local)
    row_shape = local.shape[1:]
    counts = [None] * world
    dist.all_gather_object(counts, (len(shard), local.dtype.str), group=group)
    width = int(np.prod(row_shape)) if row_shape else 1
    maxn = max(c[0] for c in counts)
    pad = np.zeros((maxn, width), dtype=local.dtype)
    pad[: len(shard)] = local.reshape(len(shard), width)
    idx = np.full(maxn, -1, dtype=np.int64)
    idx[: len(shard)] = shard
    t_rows = torch.from_numpy(pad)
    t_idx = torch.from_numpy(idx)
    rows = [torch.empty_like(t_rows) for _ in range(world)]
    idxs = [torch.empty_like(t_idx) for _ in range(world)]
    dist.all_gather(rows, t_rows, group=group)
    dist.all_gather(idxs, t_idx, group=group)
    out = np.empty((num_docs, width), dtype=local.dtype)
    seen = np.zeros(num_docs, dtype=bool)
    for r in range(world):
        n = counts[r][0]
        ii = idxs[r].numpy()[:n]
        out[ii] = rows[r].numpy()[:n]
        seen[ii] = True
    if not seen.all():
        raise RuntimeError("gather: some documents were not scored by any rank")
    return out.reshape((num_docs,) + row_shape)
