"""Float64 CPU oracle for the DSA decode path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library (``deepseek_sparse_attention_lightning_gb300``) and never imports it.

Every function follows the definition on the pages it cites, in plain numpy
float64, with library primitives (matmul, sort) as its only building blocks.
See ``dsa_oracle.py`` for the functions and for which are pinned by which
tests.
"""
from .dsa_oracle import *  # noqa: F401,F403
