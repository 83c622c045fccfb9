"""Oracle for the block-scaled FP4 routed-MoE layer: TEST INFRASTRUCTURE ONLY.

This is a plain, slow CPU statement of what the layer computes. It is written
from the web pages the method comes from and the public format specifications
they name (OCP FP8, OCP Microscaling v1.0). Floating point is fp64 unless the
definition fixes fp32: the quantiser's scale arithmetic and the router logits
that decide the top-k.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The CUDA
library shares no code with it. The only shared module is ``synthgen``, which
draws the seeded inputs and holds none of the layer's arithmetic.

Modules
-------
codecs  E2M1 / E4M3 / E8M0 decode tables and round-to-nearest-even encoders.
nvfp4   NVFP4 block quantisation, global scales and the 128x4 scale swizzle.
layout  counts, offsets without a leading 0, 128-row padded slots, capacity.
moe     router logits, softmax top-k, clamped SwiGLU and the per-token layer.
mxfp4   MXFP4 weights and the TP3 virtual-padding shard plan.

Pins: every function is checked by ``tests/test_oracle_*.py`` against something
other than itself. That means values printed on the pages (``tests/golden/``),
closed forms, exact rational brute force, library routines (``torch.topk``,
``torch.float8_e4m3fn``) or a naive second path on tiny inputs.
"""
