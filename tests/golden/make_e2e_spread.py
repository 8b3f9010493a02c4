"""Writes tests/golden/e2e_spread.txt: how far the logits of the full 32-layer
decode step move when every block's output carries a small relative rounding
error, computed with the CPU oracle alone.

The full step is the random-init Llama-3.1-8B architecture at batch 1, context
4096 (the pages' full-model decode step, summary page "전제와 한계"), drawn from
the same seeded inputs as the GPU test.  Chain A is the FP64 oracle.  Each
perturbed chain multiplies every block output elementwise by (1 + eps * n),
n ~ N(0, 1) seeded, i.e. a relative error of RMS eps per block.  eps is taken
from the kernels' arithmetic: activations enter the tensor cores as FP16
(unit roundoff 2^-11), and a value rounded to FP16 carries a relative error of
RMS about 2^-11 / sqrt(3) = 2.8e-4; 5.6e-4 doubles it.  The spread of the
logits between chains is what rounding of that size produces through 32
blocks, independent of any kernel.

Run:  python tests/golden/make_e2e_spread.py   (about 15 minutes on 8 cores)
It imports only synth/ and oracle/.
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402
from oracle.block import BlockWeightsOracle, decode_block  # noqa: E402
from oracle.kv import KVCacheOracle  # noqa: E402

EPS = (2.8e-4, 2.8e-4, 5.6e-4)     # (eps, noise seed) pairs: two seeds at 2.8e-4, one at 5.6e-4
SEEDS = (1, 2, 1)
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "e2e_spread.txt")


def rel_rms(y, ref) -> float:
    return float(np.linalg.norm(np.asarray(y) - ref) / np.linalg.norm(ref))


def main() -> None:
    wl = synth.workload("8b_full_b1_ctx4096")
    s, B, ctx, nl, V = wl.shape, wl.batch, wl.ctx, wl.layers, wl.vocab
    mt = synth.model_tensors(s, wl.config_id, V, B)
    x0 = oracle.embed(mt["emb"], mt["tokens"])
    chains = [x0.copy() for _ in range(1 + len(EPS))]
    noise = [np.random.default_rng(sd) for sd in SEEDS]
    hidden = []
    t0 = time.time()
    for li in range(nl):
        w = synth.layer_weights(s, wl.config_id, li)
        wts = BlockWeightsOracle(s, w)
        del w
        _, kf = synth.kv_history(s, wl.config_id, B, ctx, layer=li, which="k")
        _, vf = synth.kv_history(s, wl.config_id, B, ctx, layer=li, which="v")
        kc = KVCacheOracle(B, s.n_kv, ctx + 1, s.head_dim, s.hb, s.kvg)
        kc.append(kf, vf, np.zeros(B, int))
        for i, x in enumerate(chains):
            y = decode_block(s, wts, kc, x, np.full(B, ctx), write_cache=False)["out"]
            if i > 0:
                y = y * (1.0 + EPS[i - 1] * noise[i - 1].standard_normal(y.shape))
            chains[i] = y
        hidden.append([rel_rms(c, chains[0]) for c in chains[1:]])
        print(f"layer {li}: {hidden[-1]}  ({time.time() - t0:.0f} s)", flush=True)
    head = [oracle.lm_head(oracle.final_norm(c, mt["gamma_final"], s.rms_eps), mt["lm"]) for c in chains]
    logits = [rel_rms(h, head[0]) for h in head[1:]]
    with open(OUT, "w") as f:
        f.write("# Logit spread of the full 32-layer decode step (random-init Llama-3.1-8B shape, batch 1,\n")
        f.write("# context 4096) under a relative error of RMS eps on every block output; CPU oracle only.\n")
        f.write("# Written by: python tests/golden/make_e2e_spread.py\n")
        f.write("# columns: eps noise_seed final_hidden_rel_rms logits_rel_rms\n")
        for e, sd, hh, lg in zip(EPS, SEEDS, hidden[-1], logits):
            f.write(f"{e:.1e} {sd} {hh:.4e} {lg:.4e}\n")
        f.write("# hidden-state rel RMS after each layer (one column per perturbed chain):\n")
        for li, row in enumerate(hidden):
            f.write("# layer %2d " % li + " ".join(f"{v:.3e}" for v in row) + "\n")
    print(open(OUT).read())


if __name__ == "__main__":
    main()
