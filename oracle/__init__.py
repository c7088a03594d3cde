"""CPU oracle for weight-absorbed MLA decode.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may call it.  It shares no code with the CUDA library
under ``mla_absorbed_decode_gb300/``; the two meet only through the seeded
input generator, which holds none of the method's arithmetic.

Everything here is plain numpy in float64 (or pure Python for the brute-force
checks), written for a reader to check against the pages by eye:

* ``mla.py``      -- the absorbed decode definition (dense, over an FP8 E4M3
                    cache with a per-tensor scale, and over a selected top-k
                    token list), the expanded (un-absorbed) chain, the
                    LSE merge, a pure-Python brute force, the tiny full-MLA
                    example with decoupled RoPE, the FP8 projections
                    (per-tensor input quantization, bmm_fp8), and the chunked
                    expanded extend (MHA_CHUNKED_KV: chunks merged by LSE).
* ``schedule.py`` -- a restatement of the split-KV schedule rule and the
                    invariants any valid schedule must satisfy.

Parity status: every function is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py``; none is "parity unpinned".
"""
from .mla import (  # noqa: F401
    PAGE, D_LATENT, D_ROPE, D_QK,
    gather_request, visible_tokens, e4m3_value, E4M3_VALUES, dequantize_e4m3,
    decode_absorbed, decode_fp8, decode_sparse, decode_expanded, absorb_q, assemble_q, unabsorb_o,
    lse_merge, decode_bruteforce, tiny_full_mla, rope_interleaved,
    E4M3_MAX, e4m3_round, input_to_float8, bmm_fp8, absorb_q_fp8, assemble_q_fp8, unabsorb_o_fp8,
    expand_chunk, attend_chunk, extend_chunked_expanded,
)
from .schedule import schedule_reference, check_schedule  # noqa: F401
