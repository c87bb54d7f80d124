"""Marshalling helpers: host arrays (bf16 bit patterns as uint16, int32) into the
device tensors and descriptors the C ABI takes. No arithmetic of the method."""
from __future__ import annotations

import numpy as np
import torch

from . import KV, KVML, Model, ModelML

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


LAYER_NAMES = ("w_q", "w_k", "w_v", "q_norm", "k_norm", "w_o", "in_norm", "post_norm", "w_gate", "w_up", "w_down")


def model_ml_from_bits(bits: dict, shape, intermediate: int, device="cuda") -> ModelML:
    shared = {k: bf16_tensor(bits[k], device) for k in ("embed", "final_norm", "lm_head")}
    layers = [{k: bf16_tensor(l[k], device) for k in LAYER_NAMES} for l in bits["layers"]]
    return ModelML(shared, layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.vocab, intermediate,
                   shape.rms_eps, shape.rope_theta, shape.head_dim)


def kv_ml_from_docs(docs, k_pools: list, v_pools: list, device="cuda") -> KVML:
    ks = [bf16_tensor(k, device) for k in k_pools]
    vs = [bf16_tensor(v, device) for v in v_pools]
    pt = torch.from_numpy(np.ascontiguousarray(docs.page_table)).to(device)
    dl = torch.from_numpy(np.ascontiguousarray(docs.doc_len)).to(device)
    return KVML(ks, vs, pt, dl, int(docs.doc_len.max()))
