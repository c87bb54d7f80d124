"""The allocation-free trie_tree entry point (quail_classify_trie_tree_noalloc).

Some callers cannot allocate device memory: an engine that has already
claimed nearly all of the GPU's memory for its own KV pool, or a code path
where a cudaMalloc would synchronise the device mid-flight. For them the
library keeps one fixed device scratch array and this entry point places
every intermediate there. These tests call it through the C ABI and check
that two calls in a row give exactly (bit for bit) what the workspace-based
entry point gives, and, on the tiny shape, what the oracle gives.

This file is named so that pytest collects it last: if it fails, a run that
stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

import synthetic as S
from tests import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import trie_label_scoring_gb300 as Q
    Q.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def _inputs(name, ndocs):
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_from_docs
    w = S.with_docs(S.WORKLOADS[name], ndocs)
    model = C.device_model(w.shape)
    ls = S.make_labels(w, 0)
    docs = S.make_docs(w, 0)
    kv = kv_from_docs(docs)
    trie = Q.Trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
    return w, model, ls, docs, kv, trie


@pytest.mark.parametrize("name,ndocs", [("tiny-support10-4x128", 4), ("qwen3-4b-support10-256docs", 8)])
def test_noalloc_matches_workspace_entry_point_twice(name, ndocs):
    import trie_label_scoring_gb300 as Q
    w, model, ls, docs, kv, trie = _inputs(name, ndocs)
    N, M = w.num_docs, len(ls.labels)
    # reference: the existing entry point with a caller-allocated workspace
    ws = torch.empty(Q.workspace_size(model, trie, 0, N, docs.max_doc_len, Q.MODE_TRIE_TREE), dtype=torch.uint8,
                     device="cuda")
    ref_ls = torch.empty((N, M), device="cuda")
    ref_pr = torch.empty((N, M), device="cuda")
    ref_am = torch.empty((N,), dtype=torch.int32, device="cuda")
    Q.classify_trie_tree(model, kv, trie, N, ws, ref_ls, ref_pr, ref_am)
    Q.device_status()
    ref_ls, ref_pr, ref_am = ref_ls.cpu().numpy(), ref_pr.cpu().numpy(), ref_am.cpu().numpy()
    for call in range(2):  # the scratch keeps the previous call's contents
        out_ls = torch.full((N, M), float("nan"), device="cuda")
        out_pr = torch.full((N, M), float("nan"), device="cuda")
        out_am = torch.full((N,), -1, dtype=torch.int32, device="cuda")
        Q.classify_trie_tree_noalloc(model, kv, trie, N, out_ls, out_pr, out_am)
        Q.device_status()
        ls_, pr_, am_ = out_ls.cpu().numpy(), out_pr.cpu().numpy(), out_am.cpu().numpy()
        # the same kernels in the same order on the same inputs: bit-identical
        assert np.array_equal(ls_, ref_ls), f"call {call}: log scores differ from the workspace entry point"
        assert np.array_equal(pr_, ref_pr), f"call {call}: probabilities differ from the workspace entry point"
        assert np.array_equal(am_, ref_am), f"call {call}: argmax differs from the workspace entry point"
    if name.startswith("tiny"):  # and both agree with the oracle
        from oracle import scoring as OS
        from oracle.trie import build_trie
        t = build_trie(ls.labels, ls.root_token, w.shape.vocab, ls.continuation)
        L = C.oracle_layer(w.shape)
        for i in range(N):
            r = OS.trie_tree(L, *C.oracle_doc_kv(docs, i), t)
            C.check_scores(ls_[i], pr_[i], am_[i], r["logscore"], r["prob"], r["argmax"], f"doc {i} vs oracle")


def test_noalloc_rejects_calls_larger_than_the_scratch():
    import trie_label_scoring_gb300 as Q
    w, model, ls, docs, kv, trie = _inputs("qwen3-4b-support10-256docs", 8)
    big = 4096  # far more documents than 64 MiB of scratch holds at this shape
    assert Q.workspace_size(model, trie, 0, big, docs.max_doc_len, Q.MODE_TRIE_TREE) > (64 << 20)
    out = torch.empty((big, len(ls.labels)), device="cuda")
    am = torch.empty((big,), dtype=torch.int32, device="cuda")
    with pytest.raises(Q.QuailError) as e:
        Q.classify_trie_tree_noalloc(model, kv, trie, big, out, out, am)
    assert e.value.name == "QUAIL_ERR_WORKSPACE"
    assert "fixed scratch" in str(e.value)
