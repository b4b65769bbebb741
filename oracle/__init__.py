"""Plain CPU oracle of the Engram lookup layer (test infrastructure only).

This package is the slow, obviously correct statement of what the Engram hot
path computes.  It exists to check the CUDA library: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product path never calls it, and it shares no code with the
CUDA library (its only common dependency is the seeded input generators in
``workloads``, which hold none of the method's arithmetic).

Integer work is exact (Python ints / numpy uint64); floating-point work is
fp64, with bf16 rounding applied exactly where the pages place it.

Pages cited (by title):
  [P-V41]    "DeepSeek-V4.1 模型结构（5）：记忆，Engram"
  [P-LMNT]   "Engram条件记忆：DeepSeek-V4.1-Flash中196B稀疏参数N-gram哈希查表的实现原理"
  [P-O1]     "条件记忆：DeepSeek V4.1 Engram 如何用 O(1) 查表换掉一层计算"
  [P-DS4]    "ds4.c 学习笔记" — glossary entry "Engram"
  [P-DETAIL] "DeepSeek Engram 详解：把静态知识从计算里拆出来"

Modules
  layout   prime sequence, segment offsets, odd multipliers
  hashing  token map, suffix windows with pad/DEAD, multiplicative-XOR mix, row ids, history
  dequant  E4M3 x E8M0 row decode, bf16 round-to-nearest-even
  gate     wkv projection, signed-sqrt sigmoid gate, gated residual add
  shortconv the original Engram's short causal convolution on the gated value
  pipeline the five stages composed (with or without the short convolution)

Parity status: every function is pinned by tests in tests/test_oracle_*.py
except the multiplier generator, whose values cannot be pinned against a
trained checkpoint (no checkpoint exists here); see oracle.layout.
"""
from . import dequant, gate, hashing, layout, pipeline  # noqa: F401
