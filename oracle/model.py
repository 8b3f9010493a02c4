"""Full decode step: embedding, N blocks, final RMSNorm, LM head (oracle; test
infrastructure only).

The pages quote a complete Llama-3.1-8B decode step at batch 1 (summary page,
"전제와 한계") without its embedding or LM-head precision.  Readings: BF16
embedding table and LM head, FP64 residual between blocks in the oracle, final
RMSNorm z = gamma_f * rho(x) * x, logits = W_lm z.
"""
import numpy as np

from .block import decode_block, rms_factor


def embed(emb, tokens) -> np.ndarray:
    """Rows of the embedding table for the token ids, FP64 [B, H]."""
    return np.asarray(emb, dtype=np.float64)[np.asarray(tokens)]


def final_norm(x, gamma_final, eps: float) -> np.ndarray:
    """z = gamma_f * rho(x) * x with rho = (mean x^2 + eps)^-1/2, per row."""
    x = np.asarray(x, dtype=np.float64)
    return np.asarray(gamma_final, np.float64)[None, :] * rms_factor(x, eps)[:, None] * x


def lm_head(z, lm) -> np.ndarray:
    """logits[b, v] = sum_k W_lm[v, k] z[b, k]; lm is [V, H]."""
    return np.asarray(z, np.float64) @ np.asarray(lm, dtype=np.float64).T


def model_step(shape, layers, caches, emb, lm, gamma_final, tokens, pos, layer_inputs=None, final_input=None):
    """Run the full step.  ``layers``/``caches`` are per-layer oracle objects.

    ``layer_inputs`` (optional list of [B, H] arrays) teacher-forces layer l's
    input; otherwise each layer consumes the previous layer's FP64 output.
    ``final_input`` (optional [B, H]) teacher-forces the input of the final
    RMSNorm + LM head.  Returns (logits FP64 [B, V], list of per-layer results).
    """
    x = embed(emb, tokens)
    results = []
    for li, (w, c) in enumerate(zip(layers, caches)):
        xin = x if layer_inputs is None else np.asarray(layer_inputs[li], dtype=np.float64)
        r = decode_block(shape, w, c, xin, pos)
        results.append(r)
        x = r["out"]
    if final_input is not None:
        x = np.asarray(final_input, dtype=np.float64)
    logits = lm_head(final_norm(x, gamma_final, shape.rms_eps), lm)
    return logits, results
