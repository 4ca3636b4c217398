"""CPU oracle for the Hadamard-rotated Q4_0 W4A4 prefill matmul.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, CPU statement of what
the method computes, written from the engine docs page "The lean option:
ROCmFP4, ROCmI4 and Hadamard Q4_0", sections "Hadamard-rotated Q4_0: W4A4
prompt processing" and "MoE: W4A4 on the experts".  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import it.
The CUDA library never imports, links or calls anything here, and nothing here
imports the CUDA library: the two share no code.  The seeded input generators
live in their own module (``synth_inputs``) and hold none of the arithmetic.

What is pinned, and by what (tests/test_oracle_pins.py, tests/golden/):

=============================  ==============================================
function                       pinned by
=============================  ==============================================
``C_H32``                      exact rational bounds: nearest fp32 to 1/sqrt(32)
``sylvester_h32``              recursive [[H,H],[H,-H]] construction; H.H^T=32I
``fwht32``                     dense H product, exact on small integers;
                               all-ones block -> 32 e0; fp64 dot preservation
``rotate_h32``                 fp64 rotation within fp32 error bound; unit
                               vectors (hand-derived golden file)
``quantize_weights_q4_0``      round-trip bound |y-d(q-8)|<=|d|/2; signed max
                               -> code 0; fp16 scale error <= 2^-11; constant
                               and unit-vector blocks (hand-derived)
``quantize_act_int4``          round-trip bound; amax -> +-7; 2^k scale
                               invariance; hand-derived blocks
``pack_nibbles`` / unpack      exhaustive q^8 identity; brute-force bytes
``q4_0_to_aos`` / from_aos     byte-level brute force round trip
``block_partials``             brute-force integer loops
``w4a4_matmul``                brute-force fp64 loops; constant-block closed
                               form d_w d_a P = 32 alpha beta
``w4a4_matmul_id``             reduces to dense per (token, slot); brute force
``quantize_act_int8``          round-trip bound; amax -> +-127; 2^k scale
                               invariance; hand-derived blocks
``w4a8_matmul``                brute-force fp64 loops; constant-block closed
                               form d_w d_a P = 32 alpha beta
``exact_matmul``               brute-force fp64 loops
``round_bf16`` / bf16_to_f32   hand-worked ties and overflow; torch's own
                               fp32->bf16 conversion on random and edge values
``rotate_activations_bf16``    unit vectors -> bf16(+-c) (hand-derived);
                               rotate=False is bf16(x)
``rotate_importance``          closed form: the block mean (H32 entries are
                               +-1); one-hot blocks; trace preserved
``weighted_block_scale`` /     dense scans over d find nothing better;
``quantize_weights_q4_0_       Q4_0-exact blocks give error 0; never worse
weighted``                     than the plain scale; 2^k weight invariance
``pack_weights_imatrix`` /     rotated: equal to uniform weights (the pages:
``effective_importance``       on the rotated file an imatrix does nothing);
                               bad entries count as 0 before the rotation
``w4a16_matmul``               brute-force fp64 loops; Q4_0-exact weights and
                               bf16 activations reduce it to x @ w^T; constant
                               blocks: 32 d_w alpha (q - 8)
=============================  ==============================================

Every function above is pinned; none is "parity unpinned".  The informative
accuracy report (rotated vs unrotated error against ``exact_matmul``) is not a
parity target.
"""
from .hadamard import C_H32, sylvester_h32, fwht32, rotate_h32
from .quant import (
    round_half_away,
    quantize_weights_q4_0,
    quantize_act_int4,
    pack_nibbles,
    unpack_nibbles,
    act_codes_from_nibbles,
    weight_codes_from_nibbles,
    q4_0_to_aos,
    q4_0_from_aos,
    pack_weights,
    quantize_activations,
    quantize_act_int8,
    quantize_activations_int8,
    round_bf16,
    bf16_to_f32,
    rotate_activations_bf16,
    rotate_importance,
    weighted_block_scale,
    quantize_weights_q4_0_weighted,
    pack_weights_imatrix,
    effective_importance,
)
from .matmul import block_partials, w4a4_matmul, w4a4_matmul_id, w4a8_matmul, w4a16_matmul, exact_matmul

__all__ = [
    "C_H32", "sylvester_h32", "fwht32", "rotate_h32",
    "round_half_away", "quantize_weights_q4_0", "quantize_act_int4",
    "pack_nibbles", "unpack_nibbles", "act_codes_from_nibbles", "weight_codes_from_nibbles",
    "q4_0_to_aos", "q4_0_from_aos", "pack_weights", "quantize_activations",
    "quantize_act_int8", "quantize_activations_int8",
    "round_bf16", "bf16_to_f32", "rotate_activations_bf16",
    "rotate_importance", "weighted_block_scale", "quantize_weights_q4_0_weighted", "pack_weights_imatrix",
    "effective_importance",
    "block_partials", "w4a4_matmul", "w4a4_matmul_id", "w4a8_matmul", "w4a16_matmul", "exact_matmul",
]
