"""Marshalling helpers: host arrays (bf16 bit patterns as uint16, int32) into the
device tensors and descriptors the C ABI takes. No arithmetic of the method."""
from __future__ import annotations

import numpy as np
import torch

from . import KV, Model

WEIGHT_NAMES = ("embed", "w_q", "w_k", "w_v", "q_norm", "k_norm", "w_o", "in_norm", "final_norm", "lm_head")


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on `device` (bit-exact)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def model_from_bits(bits: dict, shape, device="cuda") -> Model:
    w = {k: bf16_tensor(bits[k], device) for k in WEIGHT_NAMES}
    return Model(w, shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.vocab, shape.rms_eps, shape.rope_theta,
                 shape.head_dim)


def kv_from_docs(docs, device="cuda", pin_host=False) -> KV:
    k = bf16_tensor(docs.k_pool, device)
    v = bf16_tensor(docs.v_pool, device)
    pt = torch.from_numpy(np.ascontiguousarray(docs.page_table)).to(device)
    dl = torch.from_numpy(np.ascontiguousarray(docs.doc_len)).to(device)
    return KV(k, v, pt, dl, int(docs.doc_len.max()))
