"""CPU oracle for the grouped-query attention block.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference leg may import this package. The CUDA
library and its Python binding never import it; the two share no code.

  gqa    NumPy float64 definition of the block (projections, RoPE, bf16 cache
         append, causal GQA softmax attention, output projection)
  brute  pure-Python loop restatement for tiny shapes, used to pin ``gqa``
"""
