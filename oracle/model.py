"""Full decode step: embedding, N blocks, final RMSNorm, LM head (oracle; test
infrastructure only).

The pages quote a complete Llama-3.1-8B decode step at batch 1 (summary page,
"전제와 한계") without its embedding or LM-head precision.  Readings: BF16
embedding table and LM head, FP64 residual between blocks in the oracle, final
RMSNorm z = gamma_f * rho(x) * x, logits = W_lm z.
"""
import numpy as np

from .block import decode_block, rms_factor


def model_step(shape, layers, caches, emb, lm, gamma_final, tokens, pos, layer_inputs=None):
    """Run the full step.  ``layers``/``caches`` are per-layer oracle objects.

    ``layer_inputs`` (optional list of [B, H] arrays) teacher-forces layer l's
    input; otherwise each layer consumes the previous layer's FP64 output.
    Returns (logits FP64 [B, V], list of per-layer results).
    """
    x = np.asarray(emb, dtype=np.float64)[np.asarray(tokens)]
    results = []
    for li, (w, c) in enumerate(zip(layers, caches)):
        xin = x if layer_inputs is None else np.asarray(layer_inputs[li], dtype=np.float64)
        r = decode_block(shape, w, c, xin, pos)
        results.append(r)
        x = r["out"]
    z = np.asarray(gamma_final, np.float64)[None, :] * rms_factor(x, shape.rms_eps)[:, None] * x
    logits = z @ np.asarray(lm, dtype=np.float64).T
    return logits, results
