"""Double-precision CPU oracle for exact attention (forward and backward).

TEST INFRASTRUCTURE ONLY. This package is the independent yardstick the CUDA
path is checked against. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import it; the library itself never does, and
it shares no code, table or helper with the CUDA kernels.

Everything here is IEEE double (numpy float64). Inputs are the same
bf16-rounded (or fp32) values the GPU reads, upcast exactly.

Sources (web pages on FlashAttention v1/v2/v3):
  * "FlashAttention v2相比于v1有哪些更新" (blogweb.cn), section 1: the definition
    Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V.
  * "FlashAttention技术解析" (mhpq.cn), section 2.1 (tiled pseudocode) and
    section 2.2 (online softmax with running max m and running sum l).
  * "FlashAttention v2相比于v1有哪些更新", section 3 ("Rescale操作"): the
    division by l deferred to the end of the key loop.
  * "4.3 FlashAttention-2与FlashAttention-3演进" (aiknowledge.cn), FA3 section 3:
    the forward keeps only the softmax normaliser; the backward recomputes.
  * "Flash Attention V3技术解析" (mlqm.cn), section 2.1 ("掩码处理"): causal
    blocks where the key index exceeds the query index are skipped.

`oracle.fp8` adds the FP8 (e4m3, block-scaled) quantiser and the attention of
dequantised inputs, pinned by tests/test_oracle_fp8.py.

Pins: every function here is checked by tests/test_oracle.py against things
other than itself (torch float64 scaled-dot-product attention and autograd as
an independent library routine, a pure-Python brute force, closed forms,
invariants and central finite differences). No function is "parity unpinned".
"""
from .attention import (  # noqa: F401
    forward,
    backward,
    forward_rows,
    row_statistics,
    backward_rows,
    backward_query_rows,
    tiled_forward,
)
