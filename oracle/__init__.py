"""CPU oracle for the INT4-weight / Hadamard-rotated INT4-KV decode block.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or run it.  It shares no
code with the CUDA library (no kernels, headers, tables or helpers).

The method is an encoding (INT4 codes + BF16 group scales, a block-diagonal
Hadamard rotation of the KV cache) followed by an exact computation on the
decoded values.  The oracle therefore

* re-derives every code from the FP32 inputs with the stated quantiser, taking
  each rounding decision in FP32, the precision the kernels decide in (the
  pages do not fix one), and
* evaluates the block in FP64 from those codes and scales with plain NumPy
  (a library matmul is the only primitive; no blocking, fusion or reordering).

Sources (three web pages on "FuTransformer: FP8 prefill and INT4 decode for
Llama-style inference on Hopper"):

* summary page (onedev.kr), section "어떻게 동작하나" (how it works): RMSNorm
  gain folded into the weights (W' = gamma W), row factor rho applied in the
  consumer's epilogue, direct KV placement at offset(request, head, position,
  channel).
* same page, section "무엇과 다른가" (what differs): INT4 weights and INT4 KV
  copy, group scales applied after accumulation, offset-8 nibbles, the
  block-diagonal Hadamard applied to K/V before cache quantisation and to the
  query and attention output, M=1 / skinny / split-KV decode.
* same page, section "전제와 한계" (premises and limits): GQA over 8 KV heads
  read without head expansion; round-to-nearest quantisation.

Every function states the readings it takes where the pages are silent.
"""
from .numerics import bf16_rne, bf16_bits, bf16_from_bits
from .quant import quantize_groups, dequantize_groups, nibble_decode_via_bf16
from .hadamard import sylvester, blockdiag_apply
from .rope import inv_freq, rope_apply
from .weights import quantize_weight, int4_matvec
from .kv import kv_quantize, KVCacheOracle
from .attention import attend, attend_split, merge_partials
from .block import decode_block, BlockWeightsOracle
from .model import model_step, embed, final_norm, lm_head
from .fp8 import e4m3_decode, e4m3_encode, quantize_weight_e4m3, e4m3_matvec

__all__ = [
    "bf16_rne", "bf16_bits", "bf16_from_bits",
    "quantize_groups", "dequantize_groups", "nibble_decode_via_bf16",
    "sylvester", "blockdiag_apply", "inv_freq", "rope_apply",
    "quantize_weight", "int4_matvec", "kv_quantize", "KVCacheOracle",
    "attend", "attend_split", "merge_partials",
    "decode_block", "BlockWeightsOracle", "model_step", "embed", "final_norm", "lm_head",
    "e4m3_decode", "e4m3_encode", "quantize_weight_e4m3", "e4m3_matvec",
]
