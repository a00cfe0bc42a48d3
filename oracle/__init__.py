"""CPU oracle for the DFlash draft path — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct numpy (fp64) restatement of what the DFlash
pages define: target-layer selection, context fusion, K/V injection, the
block draft forward, the fused LM-head argmax, greedy verification, and (for
the end-to-end check) a small Llama-style causal target with the greedy
speculative loop and its plain autoregressive counterpart.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library and
never imports it; the product path does not route through it.

Every function cites the passage it follows by page title and section.
Parity status of each function (what pins it) is listed in
``oracle/dflash_oracle.py``'s module docstring.
"""
from .dflash_oracle import *  # noqa: F401,F403
