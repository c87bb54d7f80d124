"""Speed-of-light cost model and method picker ("To Classify, Try a Trie Tree",
sec. 4): the oracle against the page's worked numbers and closed forms, and
the library's quail_estimate_methods against the oracle (host only)."""
import math

import numpy as np
import pytest

import synthetic as S
from oracle import cost as C
from oracle.trie import build_trie

QWEN = C.qwen3_4b_model()
HW = {"flops": 1924.5e12, "bytes": 6789.6e9}


def _support():
    w = S.WORKLOADS["tiny-support10-4x128"]
    ls = S.make_labels(w, 0)
    return ls, build_trie(ls.labels, ls.root_token, QWEN["vocab"], ls.continuation)


# ----------------------------------------------------------------- oracle pins
def test_per_token_and_head_flops_match_the_page():
    """sec. 4.2: ~7.2 GFLOP per token in projections + MLP; sec. 4.1: the head
    is 2 d V FLOP per answer position (~0.78 GFLOP for Qwen3-4B)."""
    per_tok = 2.0 * (QWEN["proj_params"] + QWEN["mlp_params"])
    assert abs(per_tok / 1e9 - 7.2) < 0.1
    assert 2.0 * QWEN["d_model"] * QWEN["vocab"] == 777_912_320


def test_extra_work_per_document_matches_the_page():
    """sec. 4.2-4.3: per document, trie_tree adds ~32 GFLOP (4 positions),
    letters ~166 GFLOP (23 instruction tokens), trie_decode ~12 GFLOP (1.5
    tokens); a 1,000-token document costs ~7 TFLOP."""
    ls, t = _support()
    b, a_dec = C.decode_shape(t)
    per_tok = 2.0 * (QWEN["proj_params"] + QWEN["mlp_params"])
    head = 2.0 * QWEN["d_model"] * QWEN["vocab"]
    tree = C.method_shape("trie_tree", 66, 10, t["n_eval"], b, QWEN["vocab"], a_dec)
    letters = C.method_shape("letters", 66, 10, t["n_eval"], b, QWEN["vocab"], a_dec)
    decode = C.method_shape("trie_decode", 66, 10, t["n_eval"], b, QWEN["vocab"], a_dec)
    assert t["n_eval"] == 4 and tree["a"] == 4
    assert abs(tree["a"] * (per_tok + head) / 1e9 - 32) < 1.0
    assert letters["q_tail"] == 89  # Table 2
    assert abs((letters["q_tail"] - 66) * per_tok / 1e9 - 166) < 3.0
    assert (b, a_dec) == (1.5, 1.5) and decode["a"] == 1.5 and decode["requests"] == 1.5
    assert abs(decode["a"] * (per_tok + head) / 1e9 - 12) < 0.5
    assert abs(1000 * per_tok / 1e12 - 7.0) < 0.3


def test_token_pass_and_kv_counts_closed_form():
    """sec. 4.1: n_tok = L1 + N (q_pre + q_tail + a), K = ceil(n_tok / C),
    R = sum (q_pre + l_i + q_tail), trie_decode (b - 1) times that."""
    docs = {"N": 3, "L1": 100 + 200 + 300, "q_pre": 2, "C": 256}
    e = C.estimate(QWEN, HW, docs, {"q_tail": 10, "a": 4.0, "v_out": 7.0, "requests": 1.0})
    assert e["n_tok"] == 600 + 3 * 16
    assert e["K"] == math.ceil(648 / 256) == 3
    assert e["R"] == 600 + 3 * 12
    assert e["B_attn"] == QWEN["kv_bytes_per_token"] * (648 + 636)
    assert e["F_head"] == 2 * QWEN["d_model"] * 7 * 3 * 4
    assert e["B_head"] == 2 * QWEN["d_model"] * 7 * 3
    d = C.estimate(QWEN, HW, docs, {"q_tail": 10, "a": 2.5, "v_out": 7.0, "requests": 2.5})
    assert d["R"] == 1.5 * 636


def test_picker_on_the_running_example():
    """sec. 4.4: trie_decode wins the running example; trie_tree wins when the
    query asks for probabilities; the three differ by a few percent because
    the prompt's prefill dominates."""
    ls, t = _support()
    b, a_dec = C.decode_shape(t)
    docs = {"N": 1000, "L1": 1000 * 100, "q_pre": 3, "C": 8192}
    best, out = C.pick(QWEN, HW, docs, 66, 10, t["n_eval"], b, False, False, a_dec)
    assert best == "trie_decode"
    ts = [out[m]["T_classify"] for m in C.METHODS]
    assert max(ts) / min(ts) < 1.15
    best, out = C.pick(QWEN, HW, docs, 66, 10, t["n_eval"], b, True, False, a_dec)
    assert best == "trie_tree" and out["trie_decode"] is None


def test_letters_wins_when_labels_share_a_long_start():
    """sec. 4.4: two labels that differ only at the end: both trie methods run
    the model on every shared token, letters does not."""
    shared = list(range(100, 120))
    t = build_trie([shared + [7], shared + [8]], 3, QWEN["vocab"])
    b, a_dec = C.decode_shape(t)
    assert (b, a_dec) == (1.0, 21.0)
    docs = {"N": 1000, "L1": 1000 * 100, "q_pre": 3, "C": 8192}
    assert C.pick(QWEN, HW, docs, 66, 2, t["n_eval"], b, False, False, a_dec)[0] == "letters"


# ------------------------------------------------------ library against oracle
def _lib_model():
    m = dict(QWEN)
    m.update(peak_flops=HW["flops"], hbm_bytes_per_s=HW["bytes"])
    return m


def _random_labels(rng, M, vocab):
    labels = set()
    while len(labels) < M:
        n = int(rng.integers(1, 6))
        labels.add(tuple(int(x) for x in rng.integers(0, 12, size=n)))
    return [list(l) for l in labels]


@pytest.mark.parametrize("seed", range(6))
def test_library_estimates_equal_the_oracle(seed):
    import trie_label_scoring_gb300 as Q
    rng = np.random.default_rng(seed)
    labels = _random_labels(rng, int(rng.integers(2, 40)), QWEN["vocab"])
    t_lib = Q.Trie(labels, 50, QWEN["vocab"])
    t = build_trie(labels, 50, QWEN["vocab"])
    b, a_dec = C.decode_shape(t)
    for need in (0, 1):
        work = dict(num_docs=int(rng.integers(1, 3000)), doc_tokens=float(rng.integers(0, 10**6)),
                    q_pre=int(rng.integers(0, 20)), q_tail=int(rng.integers(0, 200)),
                    max_pass_tokens=int(rng.integers(512, 32768)), need_probabilities=need)
        best, res = Q.estimate_methods(_lib_model(), work, t_lib)
        docs = {"N": work["num_docs"], "L1": work["doc_tokens"], "q_pre": work["q_pre"], "C": work["max_pass_tokens"]}
        obest, ores = C.pick(QWEN, HW, docs, work["q_tail"], len(labels), t["n_eval"], b, bool(need),
                             bool(t["has_prefix_labels"]), a_dec)
        assert best == obest
        keys = {"n_tok": "n_tok", "passes": "K", "kv_read_tokens": "R", "attn_bytes": "B_attn",
                "head_flops": "F_head", "head_bytes": "B_head", "t_head": "T_head", "t_proj": "T_proj",
                "t_attn": "T_attn", "t_mlp": "T_mlp", "t_classify": "T_classify"}
        for m in C.METHODS:
            assert (res[m] is None) == (ores[m] is None), m
            if res[m] is None:
                continue
            for k, ok in keys.items():
                assert res[m][k] == pytest.approx(ores[m][ok], rel=1e-12, abs=0.0), (m, k)


def test_library_rejects_bad_inputs():
    import trie_label_scoring_gb300 as Q
    t = Q.Trie([[1], [2]], 0, QWEN["vocab"])
    good = dict(num_docs=1, doc_tokens=10.0, q_pre=0, q_tail=0, max_pass_tokens=1, need_probabilities=0)
    Q.estimate_methods(_lib_model(), good, t)
    with pytest.raises(Q.QuailError):
        Q.estimate_methods(_lib_model(), dict(good, max_pass_tokens=0), t)
    with pytest.raises(Q.QuailError):
        Q.estimate_methods(dict(_lib_model(), peak_flops=0.0), good, t)
    with pytest.raises(Q.QuailError):
        Q.estimate_methods(_lib_model(), dict(good, num_docs=-1), t)
