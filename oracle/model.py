"""The layer at an answer position -- oracle (test infrastructure), float64.

What runs at a trie node ("To Classify, Try a Trie Tree", sec. 3.2 and 4.2:
each answer position is one more token through the model; its hidden state
is multiplied by the output head, sec. 4.1 "Output head"). The pages give the
model family (Qwen3-4B, d_model 2,560, vocab 151,936), Q/K normalisation with
RoPE ("Building an Ultra-High Throughput AI-SQL Engine", sec. 3.2.4 "fuse
small operations") and a BF16 head; they print no layer equations, so this
module takes the plainest reading, one decoder layer's attention block:

    x  = E[token]
    x^ = RMSNorm(x) * g_in                       RMSNorm(y) = y / sqrt(mean(y^2) + eps)
    q, k, v = x^ W_q^T, x^ W_k^T, x^ W_v^T        per head of 128
    q, k  <- per-head RMSNorm * g_q, g_k
    q, k  <- rotate-half RoPE at the absolute position (doc_len + depth)
    O   = softmax(q K^T / sqrt(128)) V            over [document KV ; own path]
    h   = x + O W_o^T
    z   = RMSNorm(h) * g_f
    logits = z W_lm^T;  log P = logits - logsumexp(logits)

GQA: query head h reads KV head h // (H_q / H_kv). The document KV is given
already normalised and rotated at positions 0..l-1.

Pinned by tests: RMSNorm closed form, RoPE against complex multiplication and
its relative-position property, attention against a textbook double loop,
log-softmax against scipy, and the flat-vs-tree equivalence.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Layer:
    """Holds the weights (widened from bf16 bits) and the layer's constants."""

    def __init__(self, bits: dict, shape, head_dtype=np.float64):
        self.d = shape.hidden
        self.hq = shape.n_q_heads
        self.hkv = shape.n_kv_heads
        self.hd = shape.head_dim
        self.V = shape.vocab
        self.eps = float(shape.rms_eps)
        self.theta = float(shape.rope_theta)
        self.embed_bits = bits["embed"]
        self.w_q = bf16_to_f64(bits["w_q"])
        self.w_k = bf16_to_f64(bits["w_k"])
        self.w_v = bf16_to_f64(bits["w_v"])
        self.w_o = bf16_to_f64(bits["w_o"])
        self.g_q = bf16_to_f64(bits["q_norm"])
        self.g_k = bf16_to_f64(bits["k_norm"])
        self.g_in = bf16_to_f64(bits["in_norm"])
        self.g_f = bf16_to_f64(bits["final_norm"])
        self.lm_bits = bits["lm_head"]
        self.head_dtype = head_dtype
        self._lm = None

    def embed(self, tok: int) -> np.ndarray:
        return bf16_to_f64(self.embed_bits[int(tok)])

    def lm_head(self) -> np.ndarray:
        """[V, d] in head_dtype (float64, or float32 to keep big vocabularies in memory)."""
        if self._lm is None:
            self._lm = bf16_to_f64(self.lm_bits).astype(self.head_dtype)
        return self._lm


def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def rope(x: np.ndarray, pos: float, theta: float) -> np.ndarray:
    """Rotate-half RoPE on the last axis (size D): pair (j, j + D/2) is rotated
    by the angle pos * theta^(-2j/D)."""
    D = x.shape[-1]
    half = D // 2
    j = np.arange(half, dtype=np.float64)
    ang = float(pos) * theta ** (-2.0 * j / D)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def token_qkv(L: Layer, tok: int, pos: int) -> tuple:
    """q [H_q, 128], k [H_kv, 128] (normalised, rotated at pos), v [H_kv, 128]."""
    x = L.embed(tok)
    xh = rms_norm(x, L.g_in, L.eps)
    q = (L.w_q @ xh).reshape(L.hq, L.hd)
    k = (L.w_k @ xh).reshape(L.hkv, L.hd)
    v = (L.w_v @ xh).reshape(L.hkv, L.hd)
    q = rope(rms_norm(q, L.g_q, L.eps), pos, L.theta)
    k = rope(rms_norm(k, L.g_k, L.eps), pos, L.theta)
    return q, k, v


def gqa_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """q [H_q, D], K and V [n, H_kv, D] -> O [H_q * D]; softmax(q.K^T/sqrt(D)) V."""
    hq, D = q.shape
    hkv = K.shape[1]
    G = hq // hkv
    out = np.empty((hq, D))
    for h in range(hq):
        g = h // G
        s = K[:, g, :] @ q[h] / np.sqrt(D)
        s = s - s.max()
        p = np.exp(s)
        p /= p.sum()
        out[h] = p @ V[:, g, :]
    return out.reshape(-1)


def output_state(L: Layer, tok: int, O: np.ndarray) -> np.ndarray:
    """z = RMSNorm(E[tok] + O W_o^T) * g_f."""
    h = L.embed(tok) + L.w_o @ O
    return rms_norm(h, L.g_f, L.eps)


def path_state(L: Layer, doc_k: np.ndarray, doc_v: np.ndarray, path_tokens: list) -> np.ndarray:
    """Hidden state z at the last token of path_tokens (root first), the path
    sitting right after the document: token j at position doc_len + j. The
    last token attends to every document token and to the whole path
    ("each node attends only to the prompt and to the nodes on its own path",
    "To Classify, Try a Trie Tree", sec. 3.2)."""
    n = doc_k.shape[0]
    ks, vs = [], []
    q = None
    for j, t in enumerate(path_tokens):
        qj, kj, vj = token_qkv(L, t, n + j)
        ks.append(kj)
        vs.append(vj)
        q = qj
    K = np.concatenate([doc_k, np.stack(ks)], axis=0)
    V = np.concatenate([doc_v, np.stack(vs)], axis=0)
    O = gqa_attention(q, K, V)
    return output_state(L, path_tokens[-1], O)


def logsumexp(x: np.ndarray) -> float:
    m = np.max(x)
    return float(m + np.log(np.sum(np.exp(x - m))))


def head_logprobs(L: Layer, z: np.ndarray) -> np.ndarray:
    """log P(token | context) over the whole vocabulary (float64)."""
    W = L.lm_head()
    logits = (W @ z.astype(W.dtype)).astype(np.float64)
    return logits - logsumexp(logits)


def head_logprobs_rows(L: Layer, Z: np.ndarray) -> np.ndarray:
    """head_logprobs for several states at once: the rows of Z [r, d] against
    the head in one product (in the head's dtype), then each row's own
    log-sum-exp in float64. Row for row the same definition as head_logprobs."""
    W = L.lm_head()
    logits = (Z.astype(W.dtype) @ W.T).astype(np.float64)
    out = np.empty_like(logits)
    for r in range(logits.shape[0]):
        out[r] = logits[r] - logsumexp(logits[r])
    return out


def sequence_logprobs(L: Layer, doc_k: np.ndarray, doc_v: np.ndarray, seq: list) -> np.ndarray:
    """Flat causal pass: the sequence seq (root first) after the document, all
    positions at once with an explicit causal mask. Returns [len(seq), V]
    log-probabilities of the next token at every position. Independent of the
    trie: used to check the tree-masked result."""
    n = doc_k.shape[0]
    T = len(seq)
    X = np.stack([L.embed(t) for t in seq])                         # [T, d]
    Xh = rms_norm(X, L.g_in, L.eps)
    Q = rms_norm((Xh @ L.w_q.T).reshape(T, L.hq, L.hd), L.g_q, L.eps)
    Kn = rms_norm((Xh @ L.w_k.T).reshape(T, L.hkv, L.hd), L.g_k, L.eps)
    Vn = (Xh @ L.w_v.T).reshape(T, L.hkv, L.hd)
    Q = np.stack([rope(Q[j], n + j, L.theta) for j in range(T)])
    Kn = np.stack([rope(Kn[j], n + j, L.theta) for j in range(T)])
    K = np.concatenate([doc_k, Kn], axis=0)                         # [n+T, Hkv, D]
    V = np.concatenate([doc_v, Vn], axis=0)
    G = L.hq // L.hkv
    mask = np.zeros((T, n + T))
    for j in range(T):
        mask[j, n + j + 1:] = -np.inf                                # causal within the sequence
    O = np.empty((T, L.hq, L.hd))
    for h in range(L.hq):
        S = Q[:, h, :] @ K[:, h // G, :].T / np.sqrt(L.hd) + mask   # [T, n+T]
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        O[:, h, :] = P @ V[:, h // G, :]
    H = X + O.reshape(T, -1) @ L.w_o.T
    Z = rms_norm(H, L.g_f, L.eps)
    W = L.lm_head()
    logits = (Z.astype(W.dtype) @ W.T).astype(np.float64)
    m = logits.max(axis=1, keepdims=True)
    return logits - (m + np.log(np.exp(logits - m).sum(axis=1, keepdims=True)))
