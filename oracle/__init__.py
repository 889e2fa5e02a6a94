"""Oracle: a plain, slow, fp64 CPU restatement of TurboQuant's KV-cache store and
decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(``cpu_baseline`` / ``--impl reference``) call it.  It shares no code, table or
constant generator with the CUDA library in ``turboquant_bit_kv_tq_gb300/``;
both sides are written from the same published description.

Sources (cited by short key in every docstring):

[Roadmap]   "From paper to practice: the TurboQuant integration roadmap for
            vLLM, SGLang and TRT-LLM", miraclefarms.github.io notes,
            2026-04-21.  §1 (core design: WHT rotation, optimal scalar
            quantiser, 1-bit QJL on the residual), §3.1-3.2 (fused store,
            fixed-grid split-KV decode, exp2), §4.2 (inverse rotation),
            §4.3 (codebook vs uniform dequant), §4.4 (masked-row and empty-split
            hazards).
[Hub]       "TurboQuant: extreme KV-cache compression for LLM inference",
            pomoai.com hub for 0xSero/turboquant.  "Technical principle",
            steps 1-5 (random orthogonal rotation, Lloyd-Max codebook for the
            Beta-distributed rotated coordinate at head_dim 128/256 and
            2/3/4 bits, QJL sign sketch of the key residual with a d x d
            random projection S, group-32 value quantisation with scale and
            zero point, bit packing 4 codes/byte at 2 bits and 2 codes/byte
            at 4 bits); "Quality cost" (cosine-similarity table).
[Paged]     "PagedAttention + TurboQuant", ithelp.ithome.com.tw article
            10406003.  "TurboQuant's core idea" (rotation keeps norms and
            geometry; MSE centroid per coordinate; 1-bit QJL on the residual
            for inner products) and "Which path vLLM takes" (store kernel
            writes the paged cache; decode reads it through the block table).
[Explainer] "TurboQuant: 3-bit KV cache", yage.ai, 2026-03-25.  The
            three-component pipeline: norm/direction split (no per-group
            metadata), MSE-optimal quantiser on the direction, residual QJL
            for key inner products.

Where the pages leave a step open this package takes the plainest reading that
the rest supports; every such reading is listed in the repository's design
notes.  Parity unpinned (nothing on the pages fixes these, so no test can pin
them to an outside value): the choice of random generator (SplitMix64 +
Box-Muller), the byte layout of a cache page, and the Lloyd initialisation path
(only its fixed point is pinned).
"""

from . import prng, codebook, rotation, quant, paged  # noqa: F401
