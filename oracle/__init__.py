"""Plain CPU oracle for the 16-token speculative-verify decode step.

TEST INFRASTRUCTURE ONLY.  This package is the slow, obviously-correct
definition that the CUDA path is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` /
``--impl reference`` legs may import it.  The product path (the C-ABI
library and its Python binding) never imports, calls or links anything here,
and this package imports nothing from the product path.

Arithmetic is float64 (numpy) except where the method fixes a storage
precision: bf16 rounding is applied exactly where the layer stores bf16
tensors, and the two places where floating point decides an integer (the
NVFP4 activation codes and the top-k expert choice) take that decision on
float32 values, the precision the kernel decides them in.

Sources, cited by page title and section:
  [newruntime]  "Muse Spark Open Ultrafast: Pushing beyond 1,000 Tokens per
                second" (newruntime.com), sections "What happened",
                "Why now".
  [ai4snews]    "Muse Spark Open decoding passes 1,000 tokens per second: one
                resident kernel per layer lifts throughput from 517 to 1,109
                tok/s" (ai4snews.wisdomeyes.cn), sections "Synopsis",
                "Interpretation", "Perspective".
  [orcarouter]  "Muse Spark Open: 1.109 token al secondo sono un cambiamento
                di kernel, non un cambiamento di modello" (orcarouter.ai),
                sections "Dove si colloca il confine del kernel",
                "Tre bollette che un kernel così grande deve pagare",
                "Su cosa vengono ancora spesi i 5,9 ms".
The pages fix the structure (62 layers, sliding window 2,048 / global
attention, top-8 of 256 experts, NVFP4 experts with bf16 layers, a pooler
before and an unpooler after the experts, an fp4 intermediate and a bf16
expert output between the two expert GEMMs).  Dimensions, norm epsilon, RoPE
theta, NVFP4 block format and the router bias law come from the workload
definitions (listed in the module docstrings where used).

Pin status: every function here is pinned by a CPU test against values or
properties that do not come from this package (hand-written tables, closed
forms, brute force on tiny inputs, invariants).  See ``tests/test_oracle_*``.
"""

from . import formats, model  # noqa: F401
