"""CPU fp64 oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package's ``smoke()`` self-check and the benchmark's CPU
baseline leg may import anything from here.  The product path (the CUDA library
and its Python binding) never imports, calls or links this package, and this
package never imports the product: the two share no code.  The only common
input is the seeded generator module, which draws inputs and holds none of the
attention arithmetic.

Contents
  attention.py  the plain definition: materialise S, softmax, multiply by V
                ("Fast Inference and Training at Scale" §6.21, standard attention);
                also the decode case (§6.1) and the merge of key-split partials.
  online.py     a tiled online-softmax pass written from the recurrence of
                "Hardware Co-Design" (FlashAttention section), in its
                per-step-normalised and deferred forms; used only to pin
                attention.py.
  codecs.py     bf16 and FP8 e4m3 decoders written from the formats' bit
                layouts, and the per-tile dequantisation of FP8 inputs.
  backward.py   the gradients dQ, dK, dV by their definition (recomputing P
                from the log-sum-exp).
  quant.py      the e4m3 encoder and the Hadamard-rotate + per-tile e4m3
                quantisation step of FlashAttention-3's FP8 path.
  pool.py       the same definitions fanned out over independent (batch,
                head) units on spawned worker processes, for whole-tensor
                checks at full size (forward heads; backward KV-head units).

Every function states the passage it follows.  Pins (tests/test_oracle.py)
check each against invariants, closed forms, brute force and library
routines.
"""
from .attention import attention, attention_rows, decode, decode_multi, decode_paged, merge_partials  # noqa: F401
from .codecs import bf16_decode, e4m3_decode, dequantize_tiles  # noqa: F401
from .online import attention_online  # noqa: F401
from .quant import e4m3_encode, rotate_quantize  # noqa: F401
from .backward import attention_backward  # noqa: F401
