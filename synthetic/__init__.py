"""Seeded synthetic inputs for trie-constrained label scoring.

This module only draws input data: weights, paged document KV, label token
lists and letter ids, all as bf16 bit patterns (uint16) or int32 arrays. It
holds none of the scoring method's arithmetic, so both the CUDA path (tests,
bench) and the CPU oracle (tests) may use it without sharing any of the
method's code.

Recipe (the shapes follow "To Classify, Try a Trie Tree", sec. 2 and 4.1,
Qwen3-4B dims: d_model 2,560, vocab 151,936):
  * numpy PCG64; SeedSequence(seed).spawn(16) gives one named sub-stream per
    tensor (see _STREAM); large tensors are drawn in fixed 4 Mi-element chunks,
    chunk j from its own child seed, so the values do not depend on the thread
    count.
  * fp32 normals N(0, std^2) rounded to bf16 with round-to-nearest-even.
  * RMSNorm gains are exactly 1.
  * Document KV lives in 16-token pages; the pool holds sum(ceil(l_i/16))
    pages whose physical order is a random permutation. Slots past a
    document's end in its last page hold bf16 NaN, so reading them shows up.
  * Label token ids: children of one trie node get distinct ids, uniform over
    [0, V); the answer token is drawn the same way.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

PAGE_SIZE = 16
BF16_NAN = np.uint16(0x7FC0)
BF16_ONE = np.uint16(0x3F80)
_CHUNK = 1 << 22

_STREAM = {
    "embed": 0, "w_q": 1, "w_k": 2, "w_v": 3, "w_o": 4, "lm_head": 5,
    "labels": 6, "doc_len": 7, "page_perm": 8, "k_pool": 9, "v_pool": 10,
    "letters": 11, "root": 12,
}


# --------------------------------------------------------------- bf16 helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    t = np.right_shift(u, 16)
    np.bitwise_and(t, 1, out=t)
    np.add(t, 0x7FFF, out=t)
    np.add(t, u, out=t)
    np.right_shift(t, 16, out=t)
    return t.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(ss: np.random.SeedSequence, n: int, std: float) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    nchunks = max(1, math.ceil(n / _CHUNK))
    seeds = ss.spawn(nchunks)

    def work(j: int) -> None:
        lo, hi = j * _CHUNK, min(n, (j + 1) * _CHUNK)
        rng = np.random.Generator(np.random.PCG64(seeds[j]))
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x)

    threads = min(nchunks, max(1, len(os.sched_getaffinity(0))))
    if threads == 1:
        for j in range(nchunks):
            work(j)
    else:
        with _cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(work, range(nchunks)))
    return out


# --------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class LayerShape:
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    vocab: int
    head_dim: int = 128
    weight_std: float = 0.02
    kv_std: float = 1.0
    rms_eps: float = 1e-6
    rope_theta: float = 1e6


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    num_docs: int
    doc_len: tuple  # (lo, hi) inclusive; lo == hi for fixed lengths
    labels: str  # "support" | "tree" | "shared" | "letters" | "join"
    num_labels: int = 10
    label_len: tuple = (1, 4)
    label_alpha: float = 0.0  # "shared": concentration of the prefix sharing


TINY = LayerShape(hidden=512, n_q_heads=8, n_kv_heads=2, vocab=8192, kv_std=0.02)
QWEN3_4B = LayerShape(hidden=2560, n_q_heads=32, n_kv_heads=8, vocab=151936)

WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-support10-4x128", TINY, 4, (128, 128), "support"),
        Workload("qwen3-4b-support10-256docs", QWEN3_4B, 256, (128, 1024), "support"),
        Workload("qwen3-4b-tree255-64x2048", QWEN3_4B, 64, (2048, 2048), "tree", 255, (1, 8)),
        Workload("qwen3-4b-letters255-64x2048", QWEN3_4B, 64, (2048, 2048), "letters", 255, (1, 1)),
        Workload("qwen3-4b-tree20-32x8192", QWEN3_4B, 32, (8192, 8192), "tree", 20, (1, 5)),
        Workload("qwen3-4b-tree5000-16x1024", QWEN3_4B, 16, (1024, 1024), "shared", 5000, (2, 10), 10.0),
        Workload("qwen3-4b-join128-64x2048", QWEN3_4B, 64, (2048, 2048), "join", 128, (3, 9)),
    ]
}



def with_docs(w: Workload, num_docs: int, doc_len: tuple | None = None) -> Workload:
    """The same workload with fewer/more documents (or other lengths): parity cases."""
    return dataclasses.replace(w, num_docs=num_docs, doc_len=doc_len or w.doc_len,
                               name=f"{w.name}[{num_docs}docs]")


def _streams(seed: int) -> list:
    return np.random.SeedSequence(seed).spawn(16)


# --------------------------------------------------------------- model
def make_model(shape: LayerShape, seed: int = 0) -> dict:
    """Random-init weights of the layer, bf16 bits, nn.Linear layout [out, in]."""
    ss = _streams(seed)
    d, hq, hkv, hd, V = shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.vocab
    s = shape.weight_std
    m = {
        "embed": _normal_bf16(ss[_STREAM["embed"]], V * d, s).reshape(V, d),
        "w_q": _normal_bf16(ss[_STREAM["w_q"]], hq * hd * d, s).reshape(hq * hd, d),
        "w_k": _normal_bf16(ss[_STREAM["w_k"]], hkv * hd * d, s).reshape(hkv * hd, d),
        "w_v": _normal_bf16(ss[_STREAM["w_v"]], hkv * hd * d, s).reshape(hkv * hd, d),
        "w_o": _normal_bf16(ss[_STREAM["w_o"]], d * hq * hd, s).reshape(d, hq * hd),
        "lm_head": _normal_bf16(ss[_STREAM["lm_head"]], V * d, s).reshape(V, d),
        "q_norm": np.full(hd, BF16_ONE, dtype=np.uint16),
        "k_norm": np.full(hd, BF16_ONE, dtype=np.uint16),
        "in_norm": np.full(d, BF16_ONE, dtype=np.uint16),
        "final_norm": np.full(d, BF16_ONE, dtype=np.uint16),
    }
    return m


# --------------------------------------------------------------- documents
@dataclasses.dataclass
class PagedDocs:
    doc_len: np.ndarray      # int32 [N]
    page_table: np.ndarray   # int32 [N, max_pages], -1 past the document
    k_pool: np.ndarray       # uint16 [P, H_kv, 16, 128]
    v_pool: np.ndarray       # uint16 [P, H_kv, 16, 128]

    @property
    def max_doc_len(self) -> int:
        return int(self.doc_len.max())

    def doc_kv(self, i: int) -> tuple:
        """Logical (K, V) of document i as bf16 bits [len, H_kv, 128] (test helper: a gather)."""
        n = int(self.doc_len[i])
        pages = self.page_table[i, : (n + PAGE_SIZE - 1) // PAGE_SIZE]
        k = self.k_pool[pages].transpose(0, 2, 1, 3).reshape(-1, self.k_pool.shape[1], self.k_pool.shape[3])[:n]
        v = self.v_pool[pages].transpose(0, 2, 1, 3).reshape(-1, self.v_pool.shape[1], self.v_pool.shape[3])[:n]
        return k, v


def make_docs(w: Workload, seed: int = 0) -> PagedDocs:
    ss = _streams(seed)
    rng = np.random.Generator(np.random.PCG64(ss[_STREAM["doc_len"]]))
    lo, hi = w.doc_len
    lens = rng.integers(lo, hi + 1, size=w.num_docs).astype(np.int32) if lo != hi else np.full(
        w.num_docs, lo, dtype=np.int32)
    npages = (lens + PAGE_SIZE - 1) // PAGE_SIZE
    total = int(npages.sum())
    prng = np.random.Generator(np.random.PCG64(ss[_STREAM["page_perm"]]))
    perm = prng.permutation(total).astype(np.int32)
    max_pages = int(npages.max())
    table = np.full((w.num_docs, max_pages), -1, dtype=np.int32)
    j = 0
    for i in range(w.num_docs):
        table[i, : npages[i]] = perm[j: j + npages[i]]
        j += npages[i]
    sh = w.shape
    per_page = sh.n_kv_heads * PAGE_SIZE * sh.head_dim
    k_pool = _normal_bf16(ss[_STREAM["k_pool"]], total * per_page, sh.kv_std).reshape(
        total, sh.n_kv_heads, PAGE_SIZE, sh.head_dim)
    v_pool = _normal_bf16(ss[_STREAM["v_pool"]], total * per_page, sh.kv_std).reshape(
        total, sh.n_kv_heads, PAGE_SIZE, sh.head_dim)
    for i in range(w.num_docs):
        r = int(lens[i]) % PAGE_SIZE
        if r:
            last = table[i, npages[i] - 1]
            k_pool[last, :, r:, :] = BF16_NAN
            v_pool[last, :, r:, :] = BF16_NAN
    return PagedDocs(lens, table, k_pool, v_pool)


# --------------------------------------------------------------- multi-layer
@dataclasses.dataclass(frozen=True)
class MLWorkload:
    """A Workload run through n_layers decoder layers (attention + SwiGLU MLP
    of width `intermediate`) instead of the single attention block."""
    name: str
    base: Workload
    n_layers: int
    intermediate: int


def _layer_streams(seed: int, layer: int, kind: int) -> list:
    return np.random.SeedSequence([seed, kind, layer]).spawn(8)


def make_model_ml(shape: LayerShape, n_layers: int, intermediate: int, seed: int = 0) -> dict:
    """Random-init weights of an n_layers model: embed, lm_head, final_norm as
    make_model, then per layer w_q, w_k, w_v, w_o, w_gate, w_up, w_down
    (~N(0, std^2), nn.Linear layout) and unit norm gains (q, k, input,
    post-attention). Layer l draws from SeedSequence([seed, 1, l])."""
    base = make_model(shape, seed)
    d, hq, hkv, hd = shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    I, st = intermediate, shape.weight_std
    layers = []
    for l in range(n_layers):
        ss = _layer_streams(seed, l, 1)
        layers.append({
            "w_q": _normal_bf16(ss[0], hq * hd * d, st).reshape(hq * hd, d),
            "w_k": _normal_bf16(ss[1], hkv * hd * d, st).reshape(hkv * hd, d),
            "w_v": _normal_bf16(ss[2], hkv * hd * d, st).reshape(hkv * hd, d),
            "w_o": _normal_bf16(ss[3], d * hq * hd, st).reshape(d, hq * hd),
            "w_gate": _normal_bf16(ss[4], I * d, st).reshape(I, d),
            "w_up": _normal_bf16(ss[5], I * d, st).reshape(I, d),
            "w_down": _normal_bf16(ss[6], d * I, st).reshape(d, I),
            "q_norm": np.full(hd, BF16_ONE, dtype=np.uint16),
            "k_norm": np.full(hd, BF16_ONE, dtype=np.uint16),
            "in_norm": np.full(d, BF16_ONE, dtype=np.uint16),
            "post_norm": np.full(d, BF16_ONE, dtype=np.uint16),
        })
    return {"embed": base["embed"], "lm_head": base["lm_head"], "final_norm": base["final_norm"], "layers": layers}


def make_docs_ml(w: Workload, n_layers: int, seed: int = 0) -> tuple:
    """Paged document KV of every layer: lengths, page table and layer 0's
    pools as make_docs; layer l >= 1 pools from SeedSequence([seed, 2, l]),
    NaN past each document's end likewise. Returns (PagedDocs of layer 0,
    [k_pool per layer], [v_pool per layer])."""
    d0 = make_docs(w, seed)
    ks, vs = [d0.k_pool], [d0.v_pool]
    sh = w.shape
    shape = d0.k_pool.shape
    n = int(np.prod(shape))
    npages = (d0.doc_len + PAGE_SIZE - 1) // PAGE_SIZE
    for l in range(1, n_layers):
        ss = _layer_streams(seed, l, 2)
        k = _normal_bf16(ss[0], n, sh.kv_std).reshape(shape)
        v = _normal_bf16(ss[1], n, sh.kv_std).reshape(shape)
        for i in range(w.num_docs):
            r = int(d0.doc_len[i]) % PAGE_SIZE
            if r:
                last = d0.page_table[i, npages[i] - 1]
                k[last, :, r:, :] = BF16_NAN
                v[last, :, r:, :] = BF16_NAN
        ks.append(k)
        vs.append(v)
    return d0, ks, vs


# --------------------------------------------------------------- labels
@dataclasses.dataclass
class LabelSet:
    labels: list            # list of lists of int token ids
    root_token: int
    continuation: np.ndarray | None  # uint8 bitmap ceil(V/8) or None

    def flat(self) -> tuple:
        """(tokens int32, offsets int64) as the C ABI takes them."""
        offs = np.zeros(len(self.labels) + 1, dtype=np.int64)
        offs[1:] = np.cumsum([len(l) for l in self.labels])
        toks = np.array([t for l in self.labels for t in l], dtype=np.int32)
        return toks, offs


def _distinct(rng, k: int, vocab: int, avoid: set | None = None) -> list:
    out: list = []
    seen = set(avoid or ())
    while len(out) < k:
        t = int(rng.integers(0, vocab))
        if t not in seen:
            seen.add(t)
            out.append(t)
    return out


# Topology of the running example (10 support-topic labels; "To Classify, Try
# a Trie Tree", sec. 2 query and sec. 3.1): token-letter sequences. Letter "M"
# stands for the "-factor" token, which continues the word "two".
SUPPORT_SHAPE = [
    "A",      # billing
    "BC",     # refund request
    "BD",     # refund status
    "EF",     # shipping delay
    "EG",     # shipping damage
    "EHI",    # shipping address change
    "JK",     # product defect
    "LMNO",   # two-factor authentication issue
    "P",      # praise
    "Q",      # other
]
SUPPORT_CONTINUATION = "M"


def support_labels(vocab: int, rng) -> LabelSet:
    letters = sorted({c for s in SUPPORT_SHAPE for c in s})
    ids = _distinct(rng, len(letters) + 1, vocab)  # all distinct (incl. the root token)
    tok = dict(zip(letters, ids[1:]))
    labels = [[tok[c] for c in s] for s in SUPPORT_SHAPE]
    bitmap = np.zeros((vocab + 7) // 8, dtype=np.uint8)
    t = tok[SUPPORT_CONTINUATION]
    bitmap[t >> 3] |= np.uint8(1 << (t & 7))
    return LabelSet(labels, ids[0], bitmap)


def tree_labels(M: int, lmin: int, lmax: int, vocab: int, rng) -> LabelSet:
    """Recursive split of M label slots. A node holding m > 1 slots branches
    into c = 2 + G children, G ~ Geometric on {0, 1, ...} with mean 0.5 (so the
    child count has mean 2.5), capped at m, and c = m one level above the
    maximum length; every child gets one slot, the other slots go to children
    uniformly at random. A node holding one slot ends in a unary tail so that
    the label's length is uniform on [max(depth, lmin), lmax]. No label is a
    prefix of another. Labels are returned in random order."""
    root = int(rng.integers(0, vocab))
    out: list = []

    def grow(prefix: list, m: int) -> None:
        depth = len(prefix)
        if m == 1:
            total = int(rng.integers(max(depth, lmin, 1), lmax + 1))
            tail = [int(t) for t in rng.integers(0, vocab, size=total - depth)]
            out.append(prefix + tail)
            return
        c = m if depth >= lmax - 1 else min(m, 2 + int(rng.geometric(2.0 / 3.0)) - 1)
        owner = np.concatenate([np.arange(c), rng.integers(0, c, size=m - c)])
        sizes = np.bincount(owner, minlength=c)
        toks = _distinct(rng, c, vocab)
        for t, s in zip(toks, sizes):
            grow(prefix + [t], int(s))

    grow([], M)
    order = rng.permutation(len(out))
    return LabelSet([out[i] for i in order], root, None)


def shared_prefix_labels(M: int, lmin: int, lmax: int, vocab: int, rng, alpha: float) -> LabelSet:
    """M labels whose lengths are uniform on [lmin, lmax], grown one at a
    time down a shared tree of prefixes. At each step of a label's walk it
    follows an existing child with probability proportional to the number of
    earlier labels that went through that child (only children that end no
    label), or opens a new child with probability alpha / (n + alpha), n the
    number of earlier labels through the node; once on a new child the rest
    of the label is new tokens. The last token always opens a new leaf, so no
    label is a prefix of another and no two labels are equal. Larger alpha
    shares less (more trie nodes). Labels are returned in generation order."""
    root = int(rng.integers(0, vocab))
    kids: list = [dict()]      # node -> {token: child}
    visits: list = [0]         # labels through the node
    open_: list = [True]       # the node ends no label, so a later label may pass through it
    out: list = []
    for _ in range(M):
        L = int(rng.integers(lmin, lmax + 1))
        node, path = 0, []
        for k in range(L):
            last = k == L - 1
            cand = [] if last else [(t, c) for t, c in kids[node].items() if open_[c]]
            n = sum(visits[c] for _, c in cand)
            u = rng.random() * (n + alpha)
            nxt = None
            if u < n:
                acc = 0
                for t, c in cand:
                    acc += visits[c]
                    if u < acc:
                        nxt = (t, c)
                        break
            if nxt is None:
                t = int(rng.integers(0, vocab))
                while t in kids[node]:
                    t = int(rng.integers(0, vocab))
                c = len(kids)
                kids.append(dict())
                visits.append(0)
                open_.append(not last)
                kids[node][t] = c
                nxt = (t, c)
            t, c = nxt
            visits[c] += 1
            path.append(t)
            node = c
        out.append(path)
    return LabelSet(out, root, None)


def make_labels(w: Workload, seed: int = 0) -> LabelSet:
    ss = _streams(seed)
    rng = np.random.Generator(np.random.PCG64(ss[_STREAM["labels"]]))
    V = w.shape.vocab
    if w.labels == "support":
        return support_labels(V, rng)
    if w.labels == "tree":
        return tree_labels(w.num_labels, w.label_len[0], w.label_len[1], V, rng)
    if w.labels == "shared":
        return shared_prefix_labels(w.num_labels, w.label_len[0], w.label_len[1], V, rng, w.label_alpha)
    if w.labels == "letters":
        ids = _distinct(rng, w.num_labels + 1, V)
        return LabelSet([[t] for t in ids[1:]], ids[0], None)
    if w.labels == "join":
        return join_partners(w.num_labels, w.label_len[0], w.label_len[1], V, rng)
    raise ValueError(w.labels)


def join_partners(n: int, lo: int, hi: int, V: int, rng) -> LabelSet:
    """Partners of a model join ("Building an Ultra-High Throughput AI-SQL
    Engine", sec. 3.2.4): after the root token, a shared instruction of 24
    tokens, the partner's own text of lo..hi tokens, and a closing answer
    token shared by all; distinct partners."""
    ids = _distinct(rng, 26, V)
    root, shared, answer = ids[0], list(ids[1:25]), ids[25]
    seen = set()
    labels = []
    while len(labels) < n:
        text = tuple(int(t) for t in rng.integers(0, V, size=int(rng.integers(lo, hi + 1))))
        if text in seen:
            continue
        seen.add(text)
        labels.append(shared + list(text) + [answer])
    return LabelSet(labels, root, None)


def make_answers(seed: int, V: int) -> tuple:
    """Token ids of the TRUE and FALSE spellings (4 each, distinct)."""
    rng = np.random.Generator(np.random.PCG64(_streams(seed)[_STREAM["letters"]]))
    ids = [int(t) for t in _distinct(rng, 8, V)]
    return ids[:4], ids[4:]


ML_WORKLOADS = {
    w.name: w
    for w in (
        MLWorkload("tiny-L3-support10-4x128", WORKLOADS["tiny-support10-4x128"], 3, 1024),
        MLWorkload("qwen3-4b-L36-support10-64docs",
                   Workload("qwen3-4b-support10-64docs", QWEN3_4B, 64, (128, 1024), "support"), 36, 9728),
    )
}


# --------------------------------------------------------------- huge label sets
@dataclasses.dataclass(frozen=True)
class ShortlistWorkload:
    """A large tree label set scored through a shortlist: the labels split
    into `groups` groups (0: ceil(sqrt K)) named by one distinct token each,
    the `beam` most likely group names kept per document, exact scores for
    the labels in them."""
    name: str
    base: Workload
    groups: int
    beam: int


def make_group_names(seed: int, G: int, name_len: int, V: int) -> list:
    """G distinct group names of name_len token ids each."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 3, G, name_len])))
    seen, out = set(), []
    while len(out) < G:
        nm = tuple(int(t) for t in rng.integers(0, V, size=name_len))
        if nm not in seen:
            seen.add(nm)
            out.append(list(nm))
    return out


SHORTLIST_WORKLOADS = {
    w.name: w
    for w in (
        ShortlistWorkload("qwen3-4b-grouped60k-16x1024",
                          Workload("qwen3-4b-tree60000-16x1024", QWEN3_4B, 16, (1024, 1024), "tree", 60000, (2, 10)),
                          0, 4),
    )
}
