"""trie_label_scoring_gb300 -- trie-constrained label scoring on one GB300.

A thin ctypes binding over libquail.so, whose C ABI is declared in
include/quail.h. Every step of the scoring path runs in the library's sm_103a
kernels; this module only marshals arguments (torch tensors -> device
pointers, Python label lists -> flat arrays). There is no CPU fallback: if the
library is missing, every call raises QuailError.

Entry points (same names as the C ABI, without the quail_ prefix):
  Trie(...)                      -> quail_trie_build / quail_trie_view / quail_trie_free
  workspace_size(...)            -> quail_workspace_size
  classify_trie_tree(...)        -> quail_classify_trie_tree
  classify_letters(...)          -> quail_classify_letters
  classify_trie_decode_step(...) -> quail_classify_trie_decode_step
  classify_trie_tree_noalloc(...) -> quail_classify_trie_tree_noalloc
  join_if(...)                   -> quail_join_if
  ModelML, KVML, workspace_size_ml(...), classify_trie_tree_ml(...)
                                 -> quail_workspace_size_ml / quail_classify_trie_tree_ml
  device_status(...)             -> quail_device_status
  set_stage_events(...)          -> quail_set_stage_events
  launch_count()                 -> quail_launch_count
  estimate_methods(...)          -> quail_estimate_methods
  Trie.grouped(...)              -> quail_trie_build_grouped
  Shortlist(...)                 -> quail_shortlist_create / quail_shortlist_groups / quail_shortlist_free
  workspace_size_shortlist(...), classify_trie_tree_shortlist(...)
                                 -> quail_workspace_size_shortlist / quail_classify_trie_tree_shortlist
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from ._build import LIB, build  # noqa: F401  (build() compiles the library in-tree)

MODE_TRIE_TREE, MODE_LETTERS, MODE_TRIE_DECODE, MODE_JOIN_IF = 0, 1, 2, 3
TRIE_FULL_DEPTH = 1
TRIE_ALL_NODES = 2
STAGES = ("prologue", "attention", "wo_norm", "head", "scoring")
# per-layer spans of classify_trie_tree_ml; layer l's span j is stage len(STAGES) + l * len(LAYER_SPANS) + j
LAYER_SPANS = ("qkv", "attention", "wo_norm", "gate_up", "silu_mul", "down")

STATUS = {
    0: "QUAIL_OK", -1: "QUAIL_ERR_INVALID_ARG", -2: "QUAIL_ERR_EMPTY_LABEL", -3: "QUAIL_ERR_DUPLICATE_LABEL",
    -4: "QUAIL_ERR_TOKEN_RANGE", -5: "QUAIL_ERR_PREFIX_LABEL_UNSUPPORTED", -6: "QUAIL_ERR_WORKSPACE",
    -7: "QUAIL_ERR_CUDA", -8: "QUAIL_ERR_DEVICE_BOUNDS", -9: "QUAIL_ERR_DEVICE_TIMEOUT",
    -10: "QUAIL_ERR_UNSUPPORTED_SHAPE",
}


class QuailError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS.get(status, str(status))


_i32p = ctypes.POINTER(ctypes.c_int32)


METHODS = ("trie_decode", "trie_tree", "letters")  # quail_method order


class CostModel(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("vocab", ctypes.c_int32), ("proj_params", ctypes.c_double),
                ("mlp_params", ctypes.c_double), ("kv_bytes_per_token", ctypes.c_double),
                ("peak_flops", ctypes.c_double), ("hbm_bytes_per_s", ctypes.c_double)]


class CostWorkload(ctypes.Structure):
    _fields_ = [("num_docs", ctypes.c_int32), ("doc_tokens", ctypes.c_double), ("q_pre", ctypes.c_int32),
                ("q_tail", ctypes.c_int32), ("max_pass_tokens", ctypes.c_int32),
                ("need_probabilities", ctypes.c_int32)]


class MethodCost(ctypes.Structure):
    _fields_ = [("runnable", ctypes.c_int32)] + [(n, ctypes.c_double) for n in (
        "q_tail", "a", "v_out", "requests", "n_tok", "passes", "kv_read_tokens", "attn_bytes", "head_flops",
        "head_bytes", "t_head", "t_proj", "t_attn", "t_mlp", "t_classify")]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_q", "w_k", "w_v", "q_norm", "k_norm", "w_o", "in_norm",
                                               "post_norm", "w_gate", "w_up", "w_down")]


class ModelMLDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("vocab", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("n_layers", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


class PagedKVML(ctypes.Structure):
    _fields_ = [("k_pools", ctypes.POINTER(ctypes.c_void_p)), ("v_pools", ctypes.POINTER(ctypes.c_void_p)),
                ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32), ("page_table", ctypes.c_void_p),
                ("max_pages", ctypes.c_int32), ("doc_len", ctypes.c_void_p), ("max_doc_len", ctypes.c_int32)]


class ModelDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("embed", ctypes.c_void_p), ("w_q", ctypes.c_void_p),
                ("w_k", ctypes.c_void_p), ("w_v", ctypes.c_void_p), ("q_norm", ctypes.c_void_p),
                ("k_norm", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("in_norm", ctypes.c_void_p),
                ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


class PagedKV(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("page_table", ctypes.c_void_p), ("max_pages", ctypes.c_int32),
                ("doc_len", ctypes.c_void_p), ("max_doc_len", ctypes.c_int32)]


class TrieCSR(ctypes.Structure):
    _fields_ = [("n_nodes", ctypes.c_int32), ("num_labels", ctypes.c_int32), ("n_eval", ctypes.c_int32),
                ("n_eval_children", ctypes.c_int32), ("max_depth", ctypes.c_int32),
                ("has_prefix_labels", ctypes.c_int32),
                ("parent", _i32p), ("depth", _i32p), ("token", _i32p), ("subtree_size", _i32p),
                ("child_offsets", _i32p), ("child_nodes", _i32p), ("child_tokens", _i32p),
                ("is_branching", ctypes.POINTER(ctypes.c_uint8)), ("subtree_labels", _i32p),
                ("node_label", _i32p), ("label_end_node", _i32p), ("label_length", _i32p),
                ("label_decide_depth", _i32p), ("eval_nodes", _i32p), ("eval_index_of_node", _i32p),
                ("eval_child_offsets", _i32p)]


# Every function the header declares, with its ctypes signature.
_SIGNATURES = {
    "quail_last_error": (ctypes.c_char_p, []),
    "quail_trie_build": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "quail_trie_view": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(TrieCSR)]),
    "quail_trie_free": (None, [ctypes.c_void_p]),
    "quail_trie_upload": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "quail_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(ModelDesc), ctypes.c_void_p, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int]),
    "quail_classify_trie_tree": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(PagedKV), ctypes.c_void_p,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "quail_classify_letters": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(PagedKV), ctypes.c_void_p,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p]),
    "quail_classify_trie_decode_step": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(PagedKV),
                                                       ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                       ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "quail_classify_trie_tree_noalloc": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(PagedKV),
                                                        ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "quail_join_if": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(PagedKV), ctypes.c_void_p,
                                     ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "quail_workspace_size_ml": (ctypes.c_size_t, [ctypes.POINTER(ModelMLDesc), ctypes.c_void_p, ctypes.c_int32,
                                                  ctypes.c_int32]),
    "quail_classify_trie_tree_ml": (ctypes.c_int, [ctypes.POINTER(ModelMLDesc), ctypes.POINTER(PagedKVML),
                                                   ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                   ctypes.c_void_p]),
    "quail_trie_build_grouped": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    "quail_shortlist_create": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    "quail_shortlist_free": (None, [ctypes.c_void_p]),
    "quail_shortlist_groups": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_void_p]),
    "quail_workspace_size_shortlist": (ctypes.c_size_t, [ctypes.POINTER(ModelDesc), ctypes.c_void_p, ctypes.c_void_p,
                                                         ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    "quail_classify_trie_tree_shortlist": (ctypes.c_int, [ctypes.POINTER(ModelDesc), ctypes.POINTER(PagedKV),
                                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t,
                                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                          ctypes.c_void_p, ctypes.c_void_p]),
    "quail_device_status": (ctypes.c_int, [ctypes.c_void_p]),
    "quail_set_stage_events": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "quail_launch_count": (ctypes.c_int32, []),
    "quail_estimate_methods": (ctypes.c_int, [ctypes.POINTER(CostModel), ctypes.POINTER(CostWorkload),
                                              ctypes.c_void_p, ctypes.POINTER(MethodCost),
                                              ctypes.POINTER(ctypes.c_int32)]),
}

# Exported for the tests only; not declared in include/quail.h.
_TEST_SIGNATURES = {
    "quail_test_set_pipeline_wait_limit": (ctypes.c_int, [ctypes.c_longlong]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libquail.so; raises QuailError when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise QuailError(-7, f"{LIB} is missing: build it with trie_label_scoring_gb300.build()")
        L = ctypes.CDLL(LIB)
        for name, (res, args) in {**_SIGNATURES, **_TEST_SIGNATURES}.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise QuailError(status, lib().quail_last_error().decode(errors="replace"))


def _ptr(t) -> int | None:
    """Device/host address of a torch tensor (or None)."""
    if t is None:
        return None
    return int(t.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ trie
def _flat_labels(labels) -> tuple:
    offs = np.zeros(len(labels) + 1, dtype=np.int64)
    offs[1:] = np.cumsum([len(l) for l in labels])
    toks = np.ascontiguousarray(np.array([t for l in labels for t in l], dtype=np.int32))
    if toks.size == 0:
        toks = np.zeros(1, dtype=np.int32)
    return toks, offs


class Trie:
    """Library-owned label trie (quail_trie_build). labels: list of token-id lists."""

    def __init__(self, labels, root_token: int, vocab: int, continuation=None, full_depth: bool = False,
                 all_nodes: bool = False, _handle=None):
        if _handle is None:
            toks, offs = _flat_labels(labels)
            cont = None if continuation is None else np.ascontiguousarray(continuation, dtype=np.uint8)
            h = ctypes.c_void_p()
            st = lib().quail_trie_build(toks.ctypes.data, offs.ctypes.data, len(labels), int(root_token), int(vocab),
                                        None if cont is None else cont.ctypes.data,
                                        (TRIE_FULL_DEPTH if full_depth else 0) | (TRIE_ALL_NODES if all_nodes else 0),
                                        ctypes.byref(h))
            _check(st)
        else:
            h = _handle
        self._h = h
        self.num_labels = len(labels)
        self.vocab = int(vocab)
        v = self.view()
        self.n_nodes, self.n_eval, self.n_eval_children = v["n_nodes"], v["n_eval"], v["n_eval_children"]
        self.has_prefix_labels = v["has_prefix_labels"]

    @property
    def handle(self):
        return self._h

    def view(self) -> dict:
        """Copies of the host CSR arrays (quail_trie_view)."""
        c = TrieCSR()
        _check(lib().quail_trie_view(self._h, ctypes.byref(c)))
        n, M, a = c.n_nodes, c.num_labels, c.n_eval

        def arr(p, k, dt=np.int32):
            return np.ctypeslib.as_array(p, shape=(k,)).astype(dt, copy=True) if k else np.zeros(0, dt)

        return {
            "n_nodes": n, "num_labels": M, "n_eval": a, "n_eval_children": c.n_eval_children,
            "max_depth": c.max_depth, "has_prefix_labels": c.has_prefix_labels,
            "parent": arr(c.parent, n), "depth": arr(c.depth, n), "token": arr(c.token, n),
            "subtree_size": arr(c.subtree_size, n), "child_offsets": arr(c.child_offsets, n + 1),
            "child_nodes": arr(c.child_nodes, n - 1), "child_tokens": arr(c.child_tokens, n - 1),
            "is_branching": arr(c.is_branching, n, np.uint8), "subtree_labels": arr(c.subtree_labels, n),
            "node_label": arr(c.node_label, n), "label_end_node": arr(c.label_end_node, M),
            "label_length": arr(c.label_length, M), "label_decide_depth": arr(c.label_decide_depth, M),
            "eval_nodes": arr(c.eval_nodes, a), "eval_index_of_node": arr(c.eval_index_of_node, n),
            "eval_child_offsets": arr(c.eval_child_offsets, a + 1),
        }

    def upload(self, stream=None) -> None:
        _check(lib().quail_trie_upload(self._h, _stream(stream)))

    @classmethod
    def grouped(cls, labels, root_token: int, vocab: int, group_names, num_groups: int = 0, continuation=None,
                full_depth: bool = False) -> tuple:
        """(trie, group_of_label) of the grouped labels (quail_trie_build_grouped):
        label m spelled as its group's name followed by the label; group_names
        lists num_groups (0: ceil(sqrt K)) token sequences of one length."""
        toks, offs = _flat_labels(labels)
        names = np.ascontiguousarray(np.array(group_names, dtype=np.int32).reshape(len(group_names), -1))
        cont = None if continuation is None else np.ascontiguousarray(continuation, dtype=np.uint8)
        gol = np.zeros(len(labels), dtype=np.int32)
        h = ctypes.c_void_p()
        _check(lib().quail_trie_build_grouped(toks.ctypes.data, offs.ctypes.data, len(labels), int(root_token),
                                              int(vocab), None if cont is None else cont.ctypes.data,
                                              TRIE_FULL_DEPTH if full_depth else 0, int(num_groups or 0),
                                              names.ctypes.data, int(names.shape[1]), ctypes.byref(h),
                                              gol.ctypes.data))
        return cls(labels, root_token, vocab, _handle=h), gol

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().quail_trie_free(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Shortlist:
    """Shortlist plan of a trie at cut depth D (quail_shortlist_create): the
    groups of labels sharing their first D tokens. Keep the trie alive."""

    def __init__(self, trie: Trie, cut_depth: int):
        h = ctypes.c_void_p()
        _check(lib().quail_shortlist_create(trie.handle, int(cut_depth), ctypes.byref(h)))
        self._h = h
        self.trie = trie
        self.cut_depth = int(cut_depth)
        self.num_groups = int(lib().quail_shortlist_groups(h, None))

    @property
    def handle(self):
        return self._h

    def group_of_label(self) -> np.ndarray:
        out = np.zeros(self.trie.num_labels, dtype=np.int32)
        lib().quail_shortlist_groups(self._h, out.ctypes.data)
        return out

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().quail_shortlist_free(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------ model and KV descriptors
class Model:
    """quail_model_desc over device bf16 tensors (kept alive by this object)."""

    def __init__(self, weights: dict, hidden: int, n_q_heads: int, n_kv_heads: int, vocab: int,
                 rms_eps: float = 1e-6, rope_theta: float = 1e6, head_dim: int = 128):
        self.weights = weights
        self.desc = ModelDesc(hidden, n_q_heads, n_kv_heads, head_dim, vocab, rms_eps, rope_theta,
                              *[_ptr(weights[k]) for k in ("embed", "w_q", "w_k", "w_v", "q_norm", "k_norm",
                                                           "w_o", "in_norm", "final_norm", "lm_head")])


class KV:
    """quail_paged_kv over device tensors: pools [P, H_kv, 16, 128] bf16, page_table [N, max_pages]
    int32, doc_len [N] int32; max_doc_len is the host-side bound."""

    def __init__(self, k_pool, v_pool, page_table, doc_len, max_doc_len: int):
        self.tensors = (k_pool, v_pool, page_table, doc_len)
        self.desc = PagedKV(_ptr(k_pool), _ptr(v_pool), int(k_pool.shape[0]), 16, _ptr(page_table),
                            int(page_table.shape[1]), _ptr(doc_len), int(max_doc_len))


class ModelML:
    """quail_model_ml_desc over device bf16 tensors: shared (embed, final_norm,
    lm_head) and per-layer dicts of w_q, w_k, w_v, q_norm, k_norm, w_o, in_norm,
    post_norm, w_gate, w_up, w_down (kept alive by this object)."""

    def __init__(self, shared: dict, layers: list, hidden: int, n_q_heads: int, n_kv_heads: int, vocab: int,
                 intermediate: int, rms_eps: float = 1e-6, rope_theta: float = 1e6, head_dim: int = 128):
        self.shared, self.layers = shared, layers
        self._lw = (LayerWeights * len(layers))(*[LayerWeights(*[_ptr(l[n]) for n, _ in LayerWeights._fields_])
                                                  for l in layers])
        self.desc = ModelMLDesc(hidden, n_q_heads, n_kv_heads, head_dim, vocab, intermediate, len(layers), rms_eps,
                                rope_theta, _ptr(shared["embed"]), _ptr(shared["final_norm"]),
                                _ptr(shared["lm_head"]), self._lw)


class KVML:
    """quail_paged_kv_ml: one K and one V pool per layer, a shared page table."""

    def __init__(self, k_pools: list, v_pools: list, page_table, doc_len, max_doc_len: int):
        self.tensors = (k_pools, v_pools, page_table, doc_len)
        self._k = (ctypes.c_void_p * len(k_pools))(*[_ptr(t) for t in k_pools])
        self._v = (ctypes.c_void_p * len(v_pools))(*[_ptr(t) for t in v_pools])
        self.desc = PagedKVML(self._k, self._v, int(k_pools[0].shape[0]), 16, _ptr(page_table),
                              int(page_table.shape[1]), _ptr(doc_len), int(max_doc_len))


# ------------------------------------------------------------------ calls
def workspace_size(model: Model, trie: Trie | None, num_letters: int, num_docs: int, max_doc_len: int,
                   mode: int) -> int:
    n = lib().quail_workspace_size(ctypes.byref(model.desc), None if trie is None else trie.handle,
                                   int(num_letters), int(num_docs), int(max_doc_len), int(mode))
    if n == 0:
        raise QuailError(-1, "workspace_size: invalid arguments")
    return int(n)


def classify_trie_tree(model: Model, kv: KV, trie: Trie, num_docs: int, workspace, label_logscore, label_prob,
                       label_argmax, stream=None) -> None:
    _check(lib().quail_classify_trie_tree(
        ctypes.byref(model.desc), ctypes.byref(kv.desc), trie.handle, int(num_docs), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(label_logscore), _ptr(label_prob), _ptr(label_argmax),
        _stream(stream)))


def classify_letters(model: Model, kv: KV, letter_tokens, root_token: int, num_docs: int, workspace,
                     letter_logprob, letter_prob, letter_argmax, stream=None) -> None:
    lt = np.ascontiguousarray(np.asarray(letter_tokens, dtype=np.int32))
    _check(lib().quail_classify_letters(
        ctypes.byref(model.desc), ctypes.byref(kv.desc), lt.ctypes.data, len(lt), int(root_token), int(num_docs),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(letter_logprob), _ptr(letter_prob),
        _ptr(letter_argmax), _stream(stream)))


def join_if(model: Model, kv: KV, partners: Trie, num_anchors: int, true_tokens, false_tokens, workspace, p_true,
            stream=None) -> None:
    """p_true [num_anchors, num_partners]: P(TRUE) at the end of every (anchor, partner) pair."""
    tok = np.ascontiguousarray(np.concatenate([np.asarray(true_tokens, dtype=np.int32),
                                               np.asarray(false_tokens, dtype=np.int32)]))
    _check(lib().quail_join_if(
        ctypes.byref(model.desc), ctypes.byref(kv.desc), partners.handle, int(num_anchors), tok.ctypes.data,
        len(true_tokens), len(false_tokens), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(p_true), _stream(stream)))


def classify_trie_decode_step(model: Model, kv: KV, trie: Trie, num_docs: int, node_cursor, label_out,
                              active_count, workspace, touched_nodes=None, stream=None) -> None:
    _check(lib().quail_classify_trie_decode_step(
        ctypes.byref(model.desc), ctypes.byref(kv.desc), trie.handle, int(num_docs), _ptr(node_cursor),
        _ptr(label_out), _ptr(active_count), _ptr(touched_nodes), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def classify_trie_tree_noalloc(model: Model, kv: KV, trie: Trie, num_docs: int, label_logscore, label_prob,
                               label_argmax, stream=None) -> None:
    """trie_tree in the library's fixed device scratch: no workspace, no device allocation."""
    _check(lib().quail_classify_trie_tree_noalloc(
        ctypes.byref(model.desc), ctypes.byref(kv.desc), trie.handle, int(num_docs), _ptr(label_logscore),
        _ptr(label_prob), _ptr(label_argmax), _stream(stream)))


def device_status(stream=None) -> None:
    _check(lib().quail_device_status(_stream(stream)))


def _test_set_pipeline_wait_limit(cycles: int) -> None:
    """Test hook (not in the public header): every pipeline wait gives up
    after `cycles` cycles; cycles <= 0 restores the default limit."""
    _check(lib().quail_test_set_pipeline_wait_limit(int(cycles)))


def set_stage_events(events) -> None:
    """events: list of 2 * n torch.cuda.Event(enable_timing=True) (entries may be None), or None to switch off."""
    if not events:
        _check(lib().quail_set_stage_events(None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(None if e is None else e.cuda_event) for e in events])
    _check(lib().quail_set_stage_events(arr, len(events) // 2))


def launch_count() -> int:
    """Kernels the last classify call on this thread launched."""
    return int(lib().quail_launch_count())


def estimate_methods(model: dict, workload: dict, trie: "Trie") -> tuple:
    """Speed-of-light estimates of trie_decode / trie_tree / letters for the
    labels of `trie` and the method the cost model picks.
    model: d_model, vocab, proj_params, mlp_params, kv_bytes_per_token,
    peak_flops, hbm_bytes_per_s; workload: num_docs, doc_tokens, q_pre, q_tail,
    max_pass_tokens, need_probabilities. Returns (best method name, {name: dict
    of the estimate, or None when the method cannot run})."""
    m = CostModel(**{k: model[k] for k, _ in CostModel._fields_})
    w = CostWorkload(**{k: int(workload[k]) if t is not ctypes.c_double else float(workload[k])
                        for k, t in CostWorkload._fields_})
    out = (MethodCost * 3)()
    best = ctypes.c_int32(-1)
    _check(lib().quail_estimate_methods(ctypes.byref(m), ctypes.byref(w), trie.handle, out, ctypes.byref(best)))
    res = {}
    for i, name in enumerate(METHODS):
        c = out[i]
        res[name] = ({k: getattr(c, k) for k, _ in MethodCost._fields_ if k != "runnable"} if c.runnable else None)
    return METHODS[best.value], res


def workspace_size_ml(model: ModelML, trie: Trie, num_docs: int, max_doc_len: int) -> int:
    n = lib().quail_workspace_size_ml(ctypes.byref(model.desc), trie.handle, int(num_docs), int(max_doc_len))
    if n == 0:
        raise QuailError(-1, "workspace_size_ml: invalid arguments")
    return int(n)


def workspace_size_shortlist(model: Model, trie: Trie, sl: Shortlist, beam: int, num_docs: int,
                             max_doc_len: int) -> int:
    n = lib().quail_workspace_size_shortlist(ctypes.byref(model.desc), trie.handle, sl.handle, int(beam),
                                             int(num_docs), int(max_doc_len))
    if n == 0:
        raise QuailError(-1, "workspace_size_shortlist: invalid arguments")
    return int(n)


def classify_trie_tree_shortlist(model: Model, kv: KV, trie: Trie, sl: Shortlist, beam: int, num_docs: int,
                                 workspace, label_logscore, label_prob, label_argmax, group_selected=None,
                                 stream=None) -> None:
    _check(lib().quail_classify_trie_tree_shortlist(
        ctypes.byref(model.desc), ctypes.byref(kv.desc), trie.handle, sl.handle, int(beam), int(num_docs),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(label_logscore), _ptr(label_prob),
        _ptr(label_argmax), None if group_selected is None else _ptr(group_selected), _stream(stream)))


def classify_trie_tree_ml(model: ModelML, kv: KVML, trie: Trie, num_docs: int, workspace, label_logscore,
                          label_prob, label_argmax, stream=None) -> None:
    _check(lib().quail_classify_trie_tree_ml(
        ctypes.byref(model.desc), ctypes.byref(kv.desc), trie.handle, int(num_docs), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(label_logscore), _ptr(label_prob), _ptr(label_argmax),
        _stream(stream)))
