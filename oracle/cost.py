"""Speed-of-light cost model and method picker -- oracle (test infrastructure).

Written from "To Classify, Try a Trie Tree", sec. 4 ("Pricing and picking a
method"): the request length r_i, the total token count n_tok, the number of
forward passes K (sec. 4.1, Table 1 and Table 2), the cached-KV reads R of
each method, the attention bytes B_attn = B_kv (W + R), the output head's
F_head / B_head / T_head (sec. 4.1 "Output head"), T_classify as the sum of the
projection, attention, MLP and head times, the expected trie_decode requests b
(sec. 4.3) and the choice of the lowest estimate among runnable methods
(sec. 4.4).

Readings where the page leaves a step open (it defers T_proj, T_attn and T_mlp
to an earlier post that is not among the pages):
  * projections and MLP follow the head's roofline form: F = 2 * P * n_tok
    FLOP and B = 2 * P * K bytes (bf16 weights streamed once per forward
    pass), T = max(F / Pi, B / beta), P = the family's weight count over all
    layers;
  * attention is bandwidth-bound: T_attn = B_attn / beta, with W = n_tok
    (every processed token writes its KV once);
  * trie_decode makes b requests per document (sec. 4.3) and runs the model
    on E[1 + depth of the node that decides the label] tokens after the
    prompt: the tokens of the path up to that branching node, forced
    single-child chains included (sec. 4.4: both trie methods pay for every
    shared token). In the running example that is 1.5 = b, the Table 2
    value. It cannot run when probabilities are requested or when a label is
    a prefix of another.

Plain float64 Python, step by step in the page's order. Pinned by
tests/test_cost_model.py against the page's worked numbers (7.2 GFLOP per
token in projections + MLP for Qwen3-4B, 0.78 GFLOP of head per answer
position, 32 / 166 / 12 GFLOP added per document by trie_tree / letters /
trie_decode, b = 1.5 for the support topics, the ~7 TFLOP of a 1,000-token
document) and against closed forms.
"""
from __future__ import annotations

import math

METHODS = ("trie_decode", "trie_tree", "letters")


def qwen3_4b_model() -> dict:
    """Qwen3-4B shapes (sec. 4.1: d_model 2,560, vocab 151,936; 36 layers,
    32 query / 8 KV heads of 128, MLP width 9,728, the model's public card)."""
    layers, d, hq, hkv, hd, ff = 36, 2560, 32, 8, 128, 9728
    return {
        "d_model": d,
        "vocab": 151936,
        "proj_params": layers * (d * (hq + 2 * hkv) * hd + hq * hd * d),
        "mlp_params": layers * 3 * d * ff,
        "kv_bytes_per_token": layers * 2 * hkv * hd * 2,
    }


def decode_shape(trie: dict) -> tuple:
    """(b, a_decode) of a trie built by oracle.trie.build_trie: b = (1/M) sum
    of the branching nodes on each label's path up to the deciding one
    (sec. 4.3); a_decode = (1/M) sum of (1 + depth of the deciding node)."""
    from oracle.trie import label_path
    M = trie["num_labels"]
    b = 0.0
    a = 0.0
    for m in range(M):
        path = label_path(trie, m)
        c, decide = 0, 0
        for k in range(len(path) - 1):
            u = path[k]
            if trie["subtree_labels"][u] <= 1:
                break
            if trie["is_branching"][u]:
                c += 1
                decide = int(trie["depth"][u])
        b += c
        a += 1 + decide
    return b / M, a / M


def method_shape(method: str, q_tail: int, num_labels: int, a_tree: float, b: float,
                 vocab: int, a_decode: float | None = None) -> dict:
    """Per-method instruction length, answer positions and output-head rows
    (sec. 4.1 Table 2; sec. 4.2: letters adds 2M + 3 instruction tokens and
    computes only the M label rows; sec. 4.3: trie_decode's b requests)."""
    if method == "trie_tree":
        return {"q_tail": q_tail, "a": float(a_tree), "v_out": float(vocab), "requests": 1.0}
    if method == "letters":
        return {"q_tail": q_tail + 2 * num_labels + 3, "a": 1.0, "v_out": float(num_labels), "requests": 1.0}
    if method == "trie_decode":
        a = float(b if a_decode is None else a_decode)
        return {"q_tail": q_tail, "a": a, "v_out": float(vocab), "requests": float(b)}
    raise ValueError(method)


def estimate(model: dict, hw: dict, docs: dict, shape: dict) -> dict:
    """SoL estimate of one method. docs: N, L1 = sum of l_i, q_pre, C;
    hw: peak bf16 FLOP/s (Pi) and HBM bytes/s (beta)."""
    N, L1, q_pre, C = docs["N"], docs["L1"], docs["q_pre"], docs["C"]
    q_tail, a = shape["q_tail"], shape["a"]
    # sec. 4.1: total tokens and forward passes
    n_tok = L1 + N * (q_pre + q_tail + a)
    K = math.ceil(n_tok / C)
    # sec. 4.1 "KV reads": prompt KV loaded once per request after the first
    prompt = L1 + N * (q_pre + q_tail)
    R = prompt if shape["requests"] <= 1.0 else (shape["requests"] - 1.0) * prompt
    W = n_tok
    B_attn = model["kv_bytes_per_token"] * (W + R)
    # sec. 4.1 "Output head"
    d = model["d_model"]
    F_head = 2.0 * d * shape["v_out"] * N * a
    B_head = 2.0 * d * shape["v_out"] * K
    T_head = max(F_head / hw["flops"], B_head / hw["bytes"])
    # projections and MLP in the head's roofline form (reading in the module docstring)
    F_proj = 2.0 * model["proj_params"] * n_tok
    T_proj = max(F_proj / hw["flops"], 2.0 * model["proj_params"] * K / hw["bytes"])
    F_mlp = 2.0 * model["mlp_params"] * n_tok
    T_mlp = max(F_mlp / hw["flops"], 2.0 * model["mlp_params"] * K / hw["bytes"])
    T_attn = B_attn / hw["bytes"]
    return {
        "n_tok": float(n_tok), "K": float(K), "R": float(R), "B_attn": B_attn,
        "F_head": F_head, "B_head": B_head, "T_head": T_head,
        "F_proj": F_proj, "F_mlp": F_mlp,
        "T_proj": T_proj, "T_attn": T_attn, "T_mlp": T_mlp,
        "T_classify": T_proj + T_attn + T_mlp + T_head,
    }


def pick(model: dict, hw: dict, docs: dict, q_tail: int, num_labels: int, a_tree: float, b: float,
         need_probabilities: bool, has_prefix_labels: bool, a_decode: float | None = None) -> tuple:
    """sec. 4.4: the runnable method with the lowest T_classify (ties: the
    order trie_decode, trie_tree, letters). Returns (method, {method: estimate
    or None when not runnable})."""
    out = {}
    for m in METHODS:
        runnable = not (m == "trie_decode" and (need_probabilities or has_prefix_labels))
        out[m] = (estimate(model, hw, docs, method_shape(m, q_tail, num_labels, a_tree, b, model["vocab"], a_decode))
                  if runnable else None)
    best = min((m for m in METHODS if out[m] is not None), key=lambda m: (out[m]["T_classify"], METHODS.index(m)))
    return best, out
