"""Plain, slow fp64 CPU oracle of the decode step -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the package smoke check and the CPU-baseline leg of the bench
may import or run anything in this directory.  The product path (the CUDA library
and its Python binding) never does, and shares no code with it: the two meet only
through the seeded inputs of the `synth` module.

What is computed (op grouping from "8 · Écrire son megakernel", §8.2, the seven
opcodes RMSNORM_QKV_ROPE, ATTENTION, ATTN_REDUCE, O_PROJ, MLP_UP_GATE, MLP_DOWN,
LM_HEAD; greedy selection of the next token, the "échantillonnage" of
"7 · AMD et le monokernel", §7.1): a Llama-style decoder -- RMSNorm, rotary
embeddings, grouped-query causal attention, SwiGLU MLP, final RMSNorm, untied LM
head, argmax.  The pages do not define the layer itself; the readings taken where
they are silent are listed in `decoder.py`'s header.

Parity pins: every function here is checked by tests/test_oracle_*.py against
closed forms, invariants, brute force on tiny inputs or library routines.
"""
from .decoder import *  # noqa: F401,F403
