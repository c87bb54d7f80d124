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


# The Qwen3-style MLP of a layer (the reading of the layer for "To Classify,
# Try a Trie Tree", sec. 4.2, "goes through the whole LLM"): SiLU on the gate
# projection, times the up projection, then the down projection, all applied
# to RMSNorm(h) * g_post where h is the state after the attention residual.
# The cases below are worked by hand with integer weights, so a swapped
# gate/up role, a missing post-norm gain or the MLP read from the wrong state
# changes the result by far more than the tolerance.
def _silu_by_hand(x: float) -> float:
    import math
    return x / (1.0 + math.exp(-x))


def _bits(a):
    return S.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _tiny_mlp_weights():
    # d = 2, width 2; every entry is exact in bf16
    return {"post_norm": np.array([2.0, 3.0]), "w_gate": np.array([[1.0, 0.0], [0.0, -1.0]]),
            "w_up": np.array([[0.0, 1.0], [1.0, 1.0]]), "w_down": np.array([[1.0, 0.0], [1.0, 1.0]])}


def _mlp_by_hand(h0: float, h1: float, eps: float, swap: bool = False, no_gain: bool = False) -> tuple:
    """down(SiLU(gate x) * up x), x = RMSNorm(h) * g_post, for the weights of
    _tiny_mlp_weights, written out scalar by scalar."""
    import math
    r = 1.0 / math.sqrt((h0 * h0 + h1 * h1) / 2.0 + eps)
    x0, x1 = h0 * r * (1.0 if no_gain else 2.0), h1 * r * (1.0 if no_gain else 3.0)
    g0, g1 = x0, -x1              # gate rows [1, 0], [0, -1]
    u0, u1 = x1, x0 + x1          # up rows   [0, 1], [1, 1]
    if swap:
        g0, g1, u0, u1 = u0, u1, g0, g1
    a0, a1 = _silu_by_hand(g0) * u0, _silu_by_hand(g1) * u1
    return a0, a0 + a1            # down rows [1, 0], [1, 1]


def test_mlp_closed_form_on_a_hand_worked_case():
    from oracle import multilayer as ML
    lw = _tiny_mlp_weights()
    h = np.array([[1.0, 1.0], [3.0, -4.0]])
    got = ML.mlp(lw, h, 0.0)
    # h = [1, 1]: RMSNorm gives [1, 1], times the gains [2, 3]: x = [2, 3];
    # gate = [2, -3], up = [3, 5]; SiLU(2) * 3 and SiLU(-3) * 5; down sums them
    a0 = 2.0 / (1.0 + np.exp(-2.0)) * 3.0
    a1 = -3.0 / (1.0 + np.exp(3.0)) * 5.0
    np.testing.assert_allclose(got[0], [a0, a0 + a1], rtol=1e-14, atol=0)
    np.testing.assert_allclose(got[1], _mlp_by_hand(3.0, -4.0, 0.0), rtol=1e-14, atol=0)


def test_mlp_pin_separates_the_plausible_mistakes():
    """The hand-worked values are far from what a swapped gate/up or a dropped
    post-norm gain would give, so the closed-form pin above catches both."""
    from oracle import multilayer as ML
    lw = _tiny_mlp_weights()
    for h in ([1.0, 1.0], [3.0, -4.0]):
        got = ML.mlp(lw, np.array([h]), 0.0)[0]
        for wrong in (_mlp_by_hand(*h, 0.0, swap=True), _mlp_by_hand(*h, 0.0, no_gain=True)):
            assert np.abs(got - np.array(wrong)).max() > 0.1


def test_layer_applies_the_mlp_to_the_state_after_attention():
    """One layer with d = 2, one head of 2 dims, W_q = W_v = 0: the query is
    zero, so the position attends uniformly to the 3 document tokens (V = 4)
    and to itself (V = 0), O = [3, 3]; with W_o = I and E[token] = [-2, -2]
    the state after attention is h = [1, 1]. The MLP must read that state,
    through its post-norm gain: H = h + mlp(h), z = RMSNorm(H)."""
    import math
    import types

    from oracle import multilayer as ML
    eps = 1e-6
    shape = types.SimpleNamespace(hidden=2, n_q_heads=1, n_kv_heads=1, head_dim=2, vocab=4, rms_eps=eps,
                                  rope_theta=1e6)
    lw = _tiny_mlp_weights()
    layer = {"w_q": _bits(np.zeros((2, 2))), "w_k": _bits([[1.0, 0.0], [0.0, 1.0]]), "w_v": _bits(np.zeros((2, 2))),
             "w_o": _bits([[1.0, 0.0], [0.0, 1.0]]), "q_norm": _bits([1.0, 1.0]), "k_norm": _bits([1.0, 1.0]),
             "in_norm": _bits([1.0, 1.0]), "post_norm": _bits(lw["post_norm"]), "w_gate": _bits(lw["w_gate"]),
             "w_up": _bits(lw["w_up"]), "w_down": _bits(lw["w_down"])}
    bits = {"embed": _bits([[-2.0, -2.0], [0.0, 0.0], [0.0, 0.0], [0.0, 0.0]]), "lm_head": _bits(np.eye(4, 2)),
            "final_norm": _bits([1.0, 1.0]), "layers": [layer]}
    md = ML.ModelML(bits, shape)
    doc_k = np.zeros((3, 1, 2))
    doc_v = np.full((3, 1, 2), 4.0)
    z = ML.sequence_states(md, [(doc_k, doc_v)], [0])[0]
    m0, m1 = _mlp_by_hand(1.0, 1.0, eps)
    H0, H1 = 1.0 + m0, 1.0 + m1
    r = 1.0 / math.sqrt((H0 * H0 + H1 * H1) / 2.0 + eps)
    np.testing.assert_allclose(z, [H0 * r, H1 * r], rtol=1e-12, atol=0)
    # the MLP read from the state before attention ([-2, -2]) gives another z
    w0, w1 = _mlp_by_hand(-2.0, -2.0, eps)
    W0, W1 = 1.0 + w0, 1.0 + w1
    rw = 1.0 / math.sqrt((W0 * W0 + W1 * W1) / 2.0 + eps)
    assert np.abs(z - np.array([W0 * rw, W1 * rw])).max() > 0.1


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
