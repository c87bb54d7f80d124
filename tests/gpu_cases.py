"""Shared set-up for the GPU parity tests and the bench: seeded synthetic
inputs moved to the device once per process, and the oracle's view of the
same inputs. Imported by tests only (and by __graft_entry__.smoke)."""
from __future__ import annotations

import functools

import numpy as np

import synthetic as S

# Tolerances (stated for the scoring path): |d log score| <= 1e-2,
# |d probability| <= 1e-3, argmax equal when the oracle's top-2 log-score gap
# exceeds 2e-2.
TOL_LOGSCORE = 1e-2
TOL_PROB = 1e-3
ARGMAX_GAP = 2e-2


@functools.lru_cache(maxsize=4)
def model_bits(shape: S.LayerShape, seed: int = 0) -> dict:
    return S.make_model(shape, seed)


@functools.lru_cache(maxsize=4)
def device_model(shape: S.LayerShape, seed: int = 0):
    from trie_label_scoring_gb300.torch_inputs import model_from_bits
    return model_from_bits(model_bits(shape, seed), shape)


@functools.lru_cache(maxsize=4)
def oracle_layer(shape: S.LayerShape, seed: int = 0):
    import oracle.model as OM
    head = np.float64 if shape.vocab <= 16384 else np.float32
    return OM.Layer(model_bits(shape, seed), shape, head_dtype=head)


def oracle_doc_kv(docs: S.PagedDocs, i: int):
    import oracle.model as OM
    k, v = docs.doc_kv(i)
    return OM.bf16_to_f64(k), OM.bf16_to_f64(v)


def check_scores(logscore_gpu, prob_gpu, argmax_gpu, logscore_ref, prob_ref, argmax_ref, where=""):
    """Element-wise comparison of one document's outputs with the oracle's."""
    ls_g = np.asarray(logscore_gpu, dtype=np.float64)
    fin = np.isfinite(logscore_ref)
    assert np.array_equal(np.isfinite(ls_g), fin), f"{where}: -inf pattern differs"
    d = np.abs(ls_g[fin] - logscore_ref[fin])
    assert d.max(initial=0.0) <= TOL_LOGSCORE, f"{where}: max |d logscore| = {d.max():.3e}"
    if prob_ref is not None:
        dp = np.abs(np.asarray(prob_gpu, dtype=np.float64) - prob_ref)
        assert dp.max(initial=0.0) <= TOL_PROB, f"{where}: max |d prob| = {dp.max():.3e}"
    srt = np.sort(logscore_ref[fin])[::-1]
    if len(srt) < 2 or srt[0] - srt[1] > ARGMAX_GAP:
        assert int(argmax_gpu) == int(argmax_ref), f"{where}: argmax {argmax_gpu} != {argmax_ref}"
    return float(d.max(initial=0.0))
