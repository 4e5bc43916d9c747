"""fp64 CPU oracle for jagged attention (JFA / GDPA).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline use it; the library never does.  It shares no code with the CUDA
path.  The arithmetic lives in ``gdpa_oracle.c`` (plain per-sample loops in
double precision); this module compiles it with gcc and marshals numpy
arrays through ctypes.

Every function follows the definition written out at the top of
``gdpa_oracle.c``, restated from "GEM Training: How Meta Doubled the
Efficiency of Its LLM-Scale Ads Foundation Model" (JFA paragraph: jagged
tensors, custom biases, asymmetric Q/KV lengths, backward; GDPA paragraph:
two matmuls with an elementwise activation in between; low-precision
paragraph: MXFP8 block scaling; SWA / block paragraph: sliding windows,
64-token blocks and the rotary-embedding backward fused into the block
kernel's epilogue).
"""
from .oracle import (  # noqa: F401
    ACT_GELU_ERF,
    ACT_GELU_TANH,
    ACT_IDENTITY,
    ACT_SILU,
    ACT_SOFTMAX,
    build,
    bwd,
    bwd_mx_operands,
    bwd_mxfp8,
    dequant_cols,
    dense_bias_offsets,
    dequant_rows,
    e4m3_decode,
    e4m3_encode,
    e8m0_nosat,
    e8m0_scale,
    fwd,
    quant_cols,
    quant_rows,
    rope_bwd,
    round_blocks_2d,
    rope_fwd,
)
