"""CPU oracle of the vision-tower encode.  TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import it; the product path never does.  See ``oracle/encode.py``;
the image preprocessing upstream of the encode (grid plan, contain resize with
bicubic filtering, gray canvas) is ``oracle/preprocess.py``.
"""
from .encode import (TOK_END, TOK_IMAGE, TOK_NEWLINE, TOK_START, attention, bits_to_f32,
                     block_tail, encode, evaluation, f32_to_bits, gelu, grid_positions, layer_norm,
                     layout, merge_unfold, merger, mlp_hidden, mm, norm, normalise, overlay, overlay_chunk, overlay_rows,
                     patchify, products, rms_norm, rope_half_vector, silu,
                     qkv_project,
                     rope, rope_angles, rope_freqs, round_bf16, softmax_rows, unpatchify,
                     vit_block)
