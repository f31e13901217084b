"""Test infrastructure: the plain CPU oracle for leak-free causal MXFP8 attention forward.

`oracle.mx` restates the OCP MX (MXFP8: E4M3 elements + E8M0 scale per block) quantisation and
decode; `oracle.attention` computes causal softmax attention on decoded operands with the
completed-block / own-block split of "[PyTorch] Add causal MXFP8 attention without future-token
leakage through V scales" (TransformerEngine PR #3865), in fp64.

Only `tests/`, the smoke check and the benchmark's CPU-baseline leg may import this package.
It shares no code with the CUDA library and never calls it.
"""
