"""The five attention workloads the library is validated and measured on.

Each entry names its shape, dtype, masking and scale; the FLOP counts follow
the usual convention for attention: 4 B Hq N^2 d for the forward (two GEMMs of
2 N^2 d each per head), halved when causal, and 2.5x that for the backward.
"""
import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "fp32" or "bf16": the element type of q, k, v, o (and grads);
    #                     "fp8e4m3": bf16 q, k, v quantised to block-scaled e4m3, bf16 o
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    backward: bool      # whether the workload includes the backward pass
    q_mult: float = 1.0  # Q is multiplied by this before rounding (logit stress run)
    sampled_rows: int = 0  # >0: check only this many seeded query/key rows per head
    block_window: int = 0  # >0: block-sparse local attention, query tile i sees key tiles i-W+1 .. i
    Nk: int = 0            # >0: key positions when they differ from N (queries = the last N of Nk)

    def block_mask(self):
        """[1, 1, T, T] booleans of the local-window block mask (None when dense)."""
        if not self.block_window:
            return None
        import numpy as np
        T = (self.N + 127) // 128
        i = np.arange(T)[:, None]
        j = np.arange(T)[None, :]
        return ((j <= i) & (j > i - self.block_window))[None, None]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops_fwd(self) -> float:
        if self.Nk:
            # exact visible (query, key) pairs: causal, query i sees keys 0 .. i + Nk - N
            if self.causal:
                off = self.Nk - self.N
                i = range(self.N)
                pairs = sum(max(0, min(self.Nk, r + off + 1)) for r in i)
            else:
                pairs = self.N * self.Nk
            return 4.0 * self.B * self.Hq * self.d * pairs
        if self.block_window:
            # visible 128 x 128 blocks: full off the diagonal, half on it (the
            # dense causal count 4 B H N^2 d / 2 is the same rule over all blocks)
            m = self.block_mask()[0, 0]
            T = m.shape[0]
            diag = int(m[range(T), range(T)].sum())
            blocks = int(m.sum()) - diag + (0.5 * diag if self.causal else diag)
            return 4.0 * self.B * self.Hq * 128 * 128 * self.d * blocks
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd

    def describe(self) -> dict:
        return {
            "workload": self.name, "dtype": self.dtype, "B": self.B, "Hq": self.Hq,
            "Hkv": self.Hkv, "N": self.N, "d": self.d, "causal": self.causal,
            "scale": self.scale, "backward": self.backward,
            **({"block_window_tiles": self.block_window} if self.block_window else {}),
            **({"Nk": self.Nk} if self.Nk else {}),
        }


WORKLOADS = {
    # fp32 single head, the smallest check: N=128, d=64, non-causal
    "fp32_h1_n128_d64": Workload("fp32_h1_n128_d64", "fp32", 1, 1, 1, 128, 64, False, False),
    # bf16 forward, 4x16 heads, N=2048, d=64, non-causal, and the same with Q x 4
    "bf16_b4_h16_n2048_d64": Workload("bf16_b4_h16_n2048_d64", "bf16", 4, 16, 16, 2048, 64, False, False),
    "bf16_b4_h16_n2048_d64_q4": Workload("bf16_b4_h16_n2048_d64_q4", "bf16", 4, 16, 16, 2048, 64, False, False, q_mult=4.0),
    # Llama-2-70B-shaped GQA layer: 64 query heads on 8 KV heads, N=4096, causal
    "bf16_gqa_b2_h64kv8_n4096_d128_causal": Workload("bf16_gqa_b2_h64kv8_n4096_d128_causal", "bf16", 2, 64, 8, 4096, 128, True, False),
    # forward + backward, 16 heads, N=8192, causal
    "bf16_h16_n8192_d128_causal_fwdbwd": Workload("bf16_h16_n8192_d128_causal_fwdbwd", "bf16", 1, 16, 16, 8192, 128, True, True),
    # long sequence forward + backward, 8 heads, N=65536, causal, 256 sampled rows per head
    "bf16_h8_n65536_d128_causal_fwdbwd": Workload("bf16_h8_n65536_d128_causal_fwdbwd", "bf16", 1, 8, 8, 65536, 128, True, True, sampled_rows=256),
    # chunked prefill: 4096 new queries at the end of 32768 positions, GQA 32 query heads on 8 KV heads, causal
    "bf16_gqa_h32kv8_nq4096_nk32768_d128_causal_fwdbwd": Workload(
        "bf16_gqa_h32kv8_nq4096_nk32768_d128_causal_fwdbwd", "bf16", 1, 32, 8, 4096, 128, True, True, Nk=32768),
    # block-sparse local attention (a window of 16 key tiles = 2048 keys, causal), 16 heads, N=32768
    "bf16_h16_n32768_d128_local16_fwdbwd": Workload("bf16_h16_n32768_d128_local16_fwdbwd", "bf16", 1, 16, 16, 32768, 128, True, True, block_window=16),
    # FP8 (e4m3, block-scaled) forward, same shape as the d = 128 fwd+bwd case; the bf16 inputs are quantised first
    "fp8_h16_n8192_d128_causal_fwd": Workload("fp8_h16_n8192_d128_causal_fwd", "fp8e4m3", 1, 16, 16, 8192, 128, True, False),
    # head dimension 256 (forward; the wide-head kernel), same N and heads as the d = 128 fwd+bwd case
    "bf16_h16_n8192_d256_causal_fwd": Workload("bf16_h16_n8192_d256_causal_fwd", "bf16", 1, 16, 16, 8192, 256, True, False),
    # head dimension 256, forward + backward (the backward in three passes over 128-row steps)
    "bf16_h16_n8192_d256_causal_fwdbwd": Workload("bf16_h16_n8192_d256_causal_fwdbwd", "bf16", 1, 16, 16, 8192, 256, True, True),
    # FP8 at head dimension 256 (the one-tile-per-CTA e4m3 kernel)
    "fp8_h16_n8192_d256_causal_fwd": Workload("fp8_h16_n8192_d256_causal_fwd", "fp8e4m3", 1, 16, 16, 8192, 256, True, False),
}

# Tolerances against the double-precision oracle on the same rounded inputs.
TOL_O_MAX = 2e-2        # max |O_gpu - O_ref|
TOL_O_MEAN = 2e-3       # mean |O_gpu - O_ref|
TOL_LSE_MAX = 1e-3      # max |LSE_gpu - LSE_ref|
TOL_GRAD_REL_FRO = 1e-2  # ||G_gpu - G_ref||_F / ||G_ref||_F per gradient tensor
