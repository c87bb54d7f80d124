"""Replica sharding across ranks (host side, CPU, gloo world size 2).

Each rank scores its own shard of documents; here the scoring of a shard is
the CPU oracle on the tiny workload (no GPU on this machine), and rank 0
checks that the gathered results equal a single-process run over all
documents, in document order."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from trie_label_scoring_gb300.replicas import partition_by_length, shard_tokens


def test_partition_covers_every_document_once_and_balances():
    rng = np.random.default_rng(0)
    lens = rng.integers(128, 1025, size=256)
    for world in (1, 2, 3, 8):
        shards = partition_by_length(lens, world)
        allidx = np.sort(np.concatenate(shards))
        assert np.array_equal(allidx, np.arange(256))
        toks = shard_tokens(lens, shards)
        # greedy longest-first: imbalance below the longest document
        assert max(toks) - min(toks) <= lens.max()


def test_partition_more_ranks_than_documents():
    shards = partition_by_length([5, 3], 4)
    assert sorted(len(s) for s in shards) == [0, 0, 1, 1]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_path):
    import torch.distributed as dist

    import synthetic as S
    from oracle import model as OM
    from oracle import scoring as OS
    from oracle.trie import build_trie
    from trie_label_scoring_gb300.replicas import gather_rows

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = S.with_docs(S.WORKLOADS["tiny-support10-4x128"], 6, (17, 130))
    docs = S.make_docs(w, 2)
    ls = S.make_labels(w, 0)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    L = OM.Layer(S.make_model(w.shape, 0), w.shape)
    shard = partition_by_length(docs.doc_len, world)[rank]
    local = []
    for i in shard:
        k, v = docs.doc_kv(int(i))
        local.append(OS.trie_tree(L, OM.bf16_to_f64(k), OM.bf16_to_f64(v), t)["logscore"])
    local = np.array(local, dtype=np.float64).reshape(len(shard), -1)
    full = gather_rows(local, shard, w.num_docs)
    if rank == 0:
        np.save(out_path, full)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_gather_equals_single_process(tmp_path):
    import synthetic as S
    from oracle import model as OM
    from oracle import scoring as OS
    from oracle.trie import build_trie
    out = str(tmp_path / "gathered.npy")
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    got = np.load(out)
    w = S.with_docs(S.WORKLOADS["tiny-support10-4x128"], 6, (17, 130))
    docs = S.make_docs(w, 2)
    ls = S.make_labels(w, 0)
    t = build_trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    L = OM.Layer(S.make_model(w.shape, 0), w.shape)
    for i in range(w.num_docs):
        k, v = docs.doc_kv(i)
        ref = OS.trie_tree(L, OM.bf16_to_f64(k), OM.bf16_to_f64(v), t)["logscore"]
        assert np.array_equal(got[i], ref)
