"""AI.IF over joined (anchor, partner) pairs -- oracle (test infrastructure).

Written from "Building an Ultra-High Throughput AI-SQL Engine", sec. 3.2.4
(one anchor, many partners: each partner attends to the anchor's KV and to
its own tokens only; the output head is restricted to the TRUE / FALSE
spellings) and the Quail "Execution" docs, "Joins" (partners do not use one
another's tokens).

Every pair is computed the plain way: the partner's tokens (root token
first) run as a flat sequence right after the anchor document, through the
layer of oracle.model, and the hidden state at its last token gives the
logits of the R answer spellings. P(TRUE) is the softmax over those R logits
summed over the TRUE spellings (reading: the answer is read as a choice among
its spellings, like letters' renormalisation). Pinned by tests/test_join.py:
the restricted softmax equals renormalising the full-vocabulary log-probs,
and p_true is 1 without FALSE spellings, 0 without TRUE ones.
"""
from __future__ import annotations

import numpy as np

from oracle import model as M


def restricted_p_true(z: np.ndarray, L: M.Layer, true_tokens, false_tokens) -> float:
    """Softmax over the answer spellings' logits z . W_lm[t], TRUE share."""
    W = L.lm_head()
    toks = list(true_tokens) + list(false_tokens)
    logits = np.array([float(W[t].astype(np.float64) @ z.astype(np.float64)) for t in toks])
    e = np.exp(logits - logits.max())
    return float(e[: len(true_tokens)].sum() / e.sum())


def join_if(L: M.Layer, doc_k, doc_v, root_token: int, partners, true_tokens, false_tokens) -> np.ndarray:
    """P(TRUE) for one anchor (its KV doc_k, doc_v) and every partner
    (token list after the root token)."""
    out = np.zeros(len(partners))
    for m, p in enumerate(partners):
        z = M.path_state(L, doc_k, doc_v, [root_token] + list(p))
        out[m] = restricted_p_true(z, L, true_tokens, false_tokens)
    return out
