"""Multi-layer trie_tree: the oracle (oracle.multilayer) against the
single-layer oracle and closed forms, and the CUDA path
(quail_classify_trie_tree_ml) against the oracle."""
import numpy as np
import pytest

import synthetic as S
from tests import gpu_cases as C


def _zero_like(a):
    return np.zeros_like(a)


def _doc_kv_layers(docs, ks, vs, i):
    """float64 (K, V) [len, H_kv, 128] of document i at every layer (a gather)."""
    import oracle.model as OM
    n = int(docs.doc_len[i])
    pages = docs.page_table[i, : (n + 15) // 16]
    out = []
    for k, v in zip(ks, vs):
        kk = k[pages].transpose(0, 2, 1, 3).reshape(-1, k.shape[1], k.shape[3])[:n]
        vv = v[pages].transpose(0, 2, 1, 3).reshape(-1, v.shape[1], v.shape[3])[:n]
        out.append((OM.bf16_to_f64(kk), OM.bf16_to_f64(vv)))
    return out


def _support_trie(vocab):
    from oracle.trie import build_trie
    ls = S.make_labels(S.WORKLOADS["tiny-support10-4x128"], 0)
    return ls, build_trie(ls.labels, ls.root_token, vocab, ls.continuation)


# ----------------------------------------------------------------- oracle pins
def test_one_layer_without_mlp_is_the_single_layer_oracle():
    from oracle import multilayer as ML
    from oracle import scoring as OS
    w = S.WORKLOADS["tiny-support10-4x128"]
    bits = S.make_model(w.shape, 0)
    layer = {k: bits[k] for k in ("w_q", "w_k", "w_v", "w_o", "q_norm", "k_norm", "in_norm")}
    layer.update(post_norm=bits["in_norm"], w_gate=np.zeros((256, w.shape.hidden), np.uint16),
                 w_up=np.zeros((256, w.shape.hidden), np.uint16), w_down=np.zeros((w.shape.hidden, 256), np.uint16))
    md = ML.ModelML({"embed": bits["embed"], "lm_head": bits["lm_head"], "final_norm": bits["final_norm"],
                     "layers": [layer]}, w.shape)
    L = C.oracle_layer(w.shape, 0)
    docs = S.make_docs(w, 0)
    ls, t = _support_trie(w.shape.vocab)
    for i in range(2):
        dk, dv = C.oracle_doc_kv(docs, i)
        a = ML.trie_tree(md, [(dk, dv)], t)["logscore"]
        b = OS.trie_tree(L, dk, dv, t)["logscore"]
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-10)


def test_a_layer_with_zero_outputs_adds_nothing():
    """W_o = 0 and W_down = 0 in the second layer: the stack equals its first layer."""
    from oracle import multilayer as ML
    mw = S.ML_WORKLOADS["tiny-L3-support10-4x128"]
    bits = S.make_model_ml(mw.base.shape, 2, mw.intermediate, 0)
    one = dict(bits, layers=bits["layers"][:1])
    two = dict(bits, layers=[bits["layers"][0], dict(bits["layers"][1], w_o=_zero_like(bits["layers"][1]["w_o"]),
                                                     w_down=_zero_like(bits["layers"][1]["w_down"]))])
    d0, ks, vs = S.make_docs_ml(mw.base, 2, 0)
    kv = _doc_kv_layers(d0, ks, vs, 1)
    seq = [7, 300, 9, 41]
    z1 = ML.sequence_states(ML.ModelML(one, mw.base.shape), kv[:1], seq)
    z2 = ML.sequence_states(ML.ModelML(two, mw.base.shape), kv, seq)
    np.testing.assert_allclose(z1, z2, rtol=0, atol=1e-12)


def test_states_are_causal():
    """A node's state from its own path equals the one inside a longer sequence."""
    from oracle import multilayer as ML
    mw = S.ML_WORKLOADS["tiny-L3-support10-4x128"]
    md = ML.ModelML(S.make_model_ml(mw.base.shape, 3, mw.intermediate, 0), mw.base.shape)
    d0, ks, vs = S.make_docs_ml(mw.base, 3, 0)
    kv = _doc_kv_layers(d0, ks, vs, 0)
    seq = [11, 22, 33, 44, 55]
    full = ML.sequence_states(md, kv, seq)
    for j in range(1, len(seq)):
        np.testing.assert_allclose(ML.sequence_states(md, kv, seq[: j + 1])[-1], full[j], rtol=0, atol=1e-12)


def test_silu_is_x_times_sigmoid():
    from scipy.special import expit

    from oracle import multilayer as ML
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(ML.silu(x), x * expit(x), rtol=1e-15, atol=1e-300)


# ------------------------------------------------------------------ GPU parity
def _run_ml(mw, docs_ml, labels, n_layers=None, seed=0):
    import torch
    import trie_label_scoring_gb300 as Q
    from trie_label_scoring_gb300.torch_inputs import kv_ml_from_docs, model_ml_from_bits
    n_layers = n_layers or mw.n_layers
    bits = S.make_model_ml(mw.base.shape, n_layers, mw.intermediate, seed)
    model = model_ml_from_bits(bits, mw.base.shape, mw.intermediate)
    d0, ks, vs = docs_ml
    kv = kv_ml_from_docs(d0, ks[:n_layers], vs[:n_layers])
    t = Q.Trie(labels.labels, labels.root_token, mw.base.shape.vocab, labels.continuation)
    N, M = len(d0.doc_len), len(labels.labels)
    ws = torch.empty(Q.workspace_size_ml(model, t, N, d0.max_doc_len), dtype=torch.uint8, device="cuda")
    lsc = torch.full((N, M), float("nan"), device="cuda")
    prob = torch.full((N, M), float("nan"), device="cuda")
    am = torch.full((N,), -1, dtype=torch.int32, device="cuda")
    Q.classify_trie_tree_ml(model, kv, t, N, ws, lsc, prob, am)
    Q.device_status()
    return bits, lsc.cpu().numpy(), prob.cpu().numpy(), am.cpu().numpy()


def _check_ml(mw, bits, docs_ml, labels, docs_idx, lsc, prob, am):
    from oracle import multilayer as ML
    from oracle.trie import build_trie
    head = np.float64 if mw.base.shape.vocab <= 16384 else np.float32
    md = ML.ModelML(bits, mw.base.shape, head_dtype=head)
    t = build_trie(labels.labels, labels.root_token, mw.base.shape.vocab, labels.continuation)
    d0, ks, vs = docs_ml
    for i in docs_idx:
        r = ML.trie_tree(md, _doc_kv_layers(d0, ks[: len(bits["layers"])], vs[: len(bits["layers"])], i), t)
        C.check_scores(lsc[i], prob[i], am[i], r["logscore"], r["prob"], r["argmax"], f"doc {i}")


@pytest.mark.gpu
def test_ml_tiny_three_layers_all_docs():
    mw = S.ML_WORKLOADS["tiny-L3-support10-4x128"]
    docs_ml = S.make_docs_ml(mw.base, mw.n_layers, 0)
    labels = S.make_labels(mw.base, 0)
    bits, lsc, prob, am = _run_ml(mw, docs_ml, labels)
    _check_ml(mw, bits, docs_ml, labels, range(4), lsc, prob, am)


@pytest.mark.gpu
def test_ml_tiny_tree_labels_tcgen05_attention():
    """60 tree labels (> 128 query rows per KV head) on ragged documents."""
    base = S.Workload("tiny-tree60-5", S.TINY, 5, (1, 500), "tree", 60, (1, 5))
    mw = S.MLWorkload("tiny-L2-tree60-5", base, 2, 512)
    docs_ml = S.make_docs_ml(base, 2, 7)
    labels = S.make_labels(base, 7)
    bits, lsc, prob, am = _run_ml(mw, docs_ml, labels)
    _check_ml(mw, bits, docs_ml, labels, range(5), lsc, prob, am)


@pytest.mark.gpu
def test_ml_qwen_shape_two_layers_sampled():
    """64 documents: 256 rows, so the gate|up projection runs without a k-split
    and SwiGLU is fused into its epilogue (the tiny cases take the k-split path)."""
    base = S.ML_WORKLOADS["qwen3-4b-L36-support10-64docs"].base
    mw = S.MLWorkload("qwen3-4b-L2-support10-64docs", base, 2, 9728)
    docs_ml = S.make_docs_ml(base, 2, 0)
    labels = S.make_labels(base, 0)
    bits, lsc, prob, am = _run_ml(mw, docs_ml, labels)
    _check_ml(mw, bits, docs_ml, labels, [0, 31, 63], lsc, prob, am)


@pytest.mark.gpu
def test_ml_full_depth_36_layers_sampled():
    """The bench workload itself: 36 Qwen3-4B-shaped layers, 64 documents;
    two documents checked against the oracle through the whole stack."""
    mw = S.ML_WORKLOADS["qwen3-4b-L36-support10-64docs"]
    docs_ml = S.make_docs_ml(mw.base, mw.n_layers, 0)
    labels = S.make_labels(mw.base, 0)
    bits, lsc, prob, am = _run_ml(mw, docs_ml, labels)
    _check_ml(mw, bits, docs_ml, labels, [0, 63], lsc, prob, am)
