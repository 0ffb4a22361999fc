"""Batch-invariant DiT AdaLN final modulation (``norm_out``) for GB300.

The operator (RL-Kernel PR 538 "final_adaln_out", section "What"):

    scale, shift = (SiLU(temb) @ W^T + b).chunk(2)      # 3072 -> 6144
    out = LayerNorm(x, eps=1e-6, no affine) * (1 + scale) + shift

with the autocast rounding points of miles_diffusion PR 108 (fp32 LayerNorm,
(1 + scale) rounded once to bf16, fp32 modulation, one bf16 store), and its
backward with token sums in a fixed 32-way tree.

The compute lives in hand-written sm_103a CUDA kernels behind a C ABI
(``include/adaln.h``, built into ``libadaln.so``).  ``binding`` is a thin
ctypes layer over it with the same entry-point names; ``synth`` draws seeded
synthetic inputs.  Importing this package loads nothing; the binding loads
the library on first use and fails loudly if it is missing.
"""

__all__ = ["binding", "synth"]
