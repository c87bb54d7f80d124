"""Multi-layer trie_tree -- oracle (test infrastructure).

"To Classify, Try a Trie Tree", sec. 3.2 and 4.2: every answer position is a
token that "goes through the whole LLM"; each trie node attends to the prompt
and to the nodes on its own path, at every layer. Here the layer stack is a
Qwen3-style decoder layer repeated n_layers times (reading: the pages name
Qwen3-4B; the MLP is SwiGLU, down(SiLU(gate x) * up x), with pre-norms), and
the document's cached K and V of every layer are inputs:

  h = E[tok]
  per layer l:  x = RMSNorm(h) g_in;  q, k, v = x W_q^T, x W_k^T, x W_v^T;
                per-head RMSNorm of q and k; RoPE at l_i + position;
                O = attention over [doc KV of layer l ; the path's own K, V]
                h = h + O W_o^T
                h = h + W_down (SiLU(RMSNorm(h) g_post W_gate^T) * (RMSNorm(h) g_post W_up^T))
  z = RMSNorm(h) g_f;  log-probs = log_softmax(z W_lm^T)

Plain float64 numpy, a flat causal pass over each label's path (root first),
so every node's state is computed without the trie (the path through it is a
prefix of the label's path). Pinned by tests/test_multilayer.py: one layer
with zero MLP weights equals the single-layer oracle (oracle.model); the
trie's scores equal per-label flat sequences; the MLP against its closed form.
"""
from __future__ import annotations

import numpy as np

from oracle import model as M
from oracle import scoring as OS
from oracle.trie import children_of


class ModelML:
    """Weights of an n-layer model (bf16 bits widened exactly to float64)."""

    def __init__(self, bits: dict, shape, head_dtype=np.float64):
        self.d, self.hq, self.hkv, self.hd, self.V = (shape.hidden, shape.n_q_heads, shape.n_kv_heads,
                                                      shape.head_dim, shape.vocab)
        self.eps = float(shape.rms_eps)
        self.theta = float(shape.rope_theta)
        self.embed_bits = bits["embed"]
        self.lm_bits = bits["lm_head"]
        self.g_f = M.bf16_to_f64(bits["final_norm"])
        self.layers = [{k: M.bf16_to_f64(v) for k, v in lb.items()} for lb in bits["layers"]]
        self.head_dtype = head_dtype
        self._lm = None

    def embed(self, tok: int) -> np.ndarray:
        return M.bf16_to_f64(self.embed_bits[int(tok)])

    def lm_head(self) -> np.ndarray:
        if self._lm is None:
            self._lm = M.bf16_to_f64(self.lm_bits).astype(self.head_dtype)
        return self._lm


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def mlp(lw: dict, h: np.ndarray, eps: float) -> np.ndarray:
    """down(SiLU(gate x) * up x), x = RMSNorm(h) g_post (rows of h)."""
    x = M.rms_norm(h, lw["post_norm"], eps)
    return (silu(x @ lw["w_gate"].T) * (x @ lw["w_up"].T)) @ lw["w_down"].T


def sequence_states(md: ModelML, doc_kv: list, seq: list) -> np.ndarray:
    """Final-norm states z [T, d] of the flat causal sequence seq (root
    first) right after the document; doc_kv[l] = (K, V) of layer l, float64
    [n, H_kv, 128]. Position j sits at n + j and attends to the document and
    to seq[: j + 1]."""
    n = doc_kv[0][0].shape[0]
    T = len(seq)
    H = np.stack([md.embed(t) for t in seq])  # [T, d]
    for l, lw in enumerate(md.layers):
        X = M.rms_norm(H, lw["in_norm"], md.eps)
        Q = M.rms_norm((X @ lw["w_q"].T).reshape(T, md.hq, md.hd), lw["q_norm"], md.eps)
        Kn = M.rms_norm((X @ lw["w_k"].T).reshape(T, md.hkv, md.hd), lw["k_norm"], md.eps)
        Vn = (X @ lw["w_v"].T).reshape(T, md.hkv, md.hd)
        Q = np.stack([M.rope(Q[j], n + j, md.theta) for j in range(T)])
        Kn = np.stack([M.rope(Kn[j], n + j, md.theta) for j in range(T)])
        dk, dv = doc_kv[l]
        O = np.empty((T, md.hq * md.hd))
        for j in range(T):
            K = np.concatenate([dk, Kn[: j + 1]], axis=0)
            V = np.concatenate([dv, Vn[: j + 1]], axis=0)
            O[j] = M.gqa_attention(Q[j], K, V)
        H = H + O @ lw["w_o"].T
        H = H + mlp(lw, H, md.eps)
    return M.rms_norm(H, md.g_f, md.eps)


def logprobs(md: ModelML, z: np.ndarray) -> np.ndarray:
    """log P(token | context) over the vocabulary for one state z."""
    W = md.lm_head()
    logits = (W @ z.astype(W.dtype)).astype(np.float64)
    return logits - M.logsumexp(logits)


def trie_tree(md: ModelML, doc_kv: list, trie: dict) -> dict:
    """trie_tree scores of one document through the whole layer stack: each
    evaluated node's state comes from a flat pass over a label path through it."""
    tok = trie["token"]
    states = {}
    for m in range(trie["num_labels"]):
        path = [int(trie["label_end_node"][m])]
        while path[-1] != 0:
            path.append(int(trie["parent"][path[-1]]))
        path = path[::-1]
        need = [k for k, u in enumerate(path) if trie["eval_index_of_node"][u] >= 0 and u not in states]
        if not need:
            continue
        Z = sequence_states(md, doc_kv, [int(tok[u]) for u in path[: max(need) + 1]])
        for k in need:
            states[path[k]] = Z[k]
    rows = {}
    for e in trie["eval_nodes"]:
        e = int(e)
        lp = logprobs(md, states[e])
        rows[e] = {int(tok[c]): float(lp[tok[c]]) for c in children_of(trie, e)}
    ls = OS.logscores_from_table(trie, lambda u, t: rows[u][t])
    prob, am = OS.normalise(ls)
    return {"logscore": ls, "prob": prob, "argmax": am, "rows": rows}
