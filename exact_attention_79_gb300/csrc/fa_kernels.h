// Host-visible interface between the C ABI (fa_api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

struct FwdParams {
  float* lse;                      // [B*Hq*N] natural-log logsumexp
  unsigned* status;                // device status word
  int N, Hq, Hkv, BH;              // N: query positions; BH = B*Hq
  int Nk;                          // key positions (== N unless the caller passes another length)
  int causal_off;                  // Nk - N: key j visible to query i iff j <= i + causal_off (when causal)
  int num_pairs;                   // CTAs per head (set by launch_fwd: 2 query tiles per CTA for bf16, 1 for fp32)
  int causal;
  float scale_log2;                // scale * log2(e)
  unsigned long long timeout_ns;   // bound on every wait inside the kernel
  // optional block mask (bf16 only): byte (b, h, i, j) at mask[b*mask_sb + h*mask_sh + i*mask_nt + j]
  // says whether query tile i may see key tile j (128 x 128 tiles); nullptr = dense
  const unsigned char* mask;
  long long mask_sb, mask_sh;
  int mask_nt;                     // tiles per row = ceil(N / 128)
  int test_stall;                  // 1: the issuer first waits on a barrier nothing arrives on (timeout test)
  int head_group;                  // wide-head forward: heads scheduled together (set by launch_fwd_wide)
  // FP8 forward: fp32 scales of the e4m3 inputs; Q and K one per 64-row block
  // ([BH, ceil(N/64)], [BHkv, ceil(N/64)]), V one per column ([BHkv, d])
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int head_dim;                    // FP8 forward: d (64 runs in the d = 128 kernel, columns past d zero)
  unsigned long long* clock_acc;   // [2] SM cycles and ns of every CTA's lifetime, summed (fwd_kernel); may be null
};
constexpr int kMaskMaxTiles = 1024;  // block-mask rows up to 1024 tiles (N <= 131072)

// dtype_bytes: 2 = bf16 (tensor-core kind::f16), 4 = fp32 (kind::tf32).
cudaError_t launch_fwd(int dtype_bytes, int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mo, FwdParams p, cudaStream_t stream);

// bf16, d in (64, 128], no block mask: clusters of two CTAs (four query tiles)
// whose MMAs run as cta_group::2 pairs; mk64 is the K map with 64-row boxes
// (each CTA loads half of every K tile), mv the usual V map.
cudaError_t launch_fwd_pair(const CUtensorMap& mq, const CUtensorMap& mk64, const CUtensorMap& mv,
                            const CUtensorMap& mo, FwdParams p, cudaStream_t stream);

// Head dims 136..256 (bf16, dense): one 128-row query tile per CTA; the V
// map has 64-row boxes (the kernel stages V in 64-key halves).
cudaError_t launch_fwd_wide(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mo, const FwdParams& p, cudaStream_t stream);

// FP8 (e4m3) path, d a multiple of 16 up to 256. Quantisers: rows of x [BH, N, d] bf16 -> codes
// [BH, N, d] and one scale per 64-row block; V [BH, N, d] bf16 -> V^T codes
// [BH, d, NP] (NP = N rounded up to 128, zero codes past N) and one scale per
// column (`scales` doubles as scratch for the column maxima). The forward
// reads Q, K codes (maps with 128-byte rows), V^T codes (map over [BH, d, NP])
// and writes bf16 O and the LSE.
cudaError_t launch_fp8_quant_rows(const void* x, void* out, float* scales, int BH, int N, int d,
                                  cudaStream_t stream);
cudaError_t launch_fp8_quant_v(const void* v, void* vt, float* scales, int BH, int N, int d, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mvt,
                           const CUtensorMap& mo, FwdParams p, cudaStream_t stream);
// The same computation for d in (128, 256]: one 128-row query tile per CTA,
// Q / K maps with 128-byte boxes read at x = 0 and 128, the V^T map's 128-row
// boxes at y = 0 and 128 (rows past d read as zeros).
cudaError_t launch_fwd_fp8_wide(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mvt,
                                const CUtensorMap& mo, FwdParams p, cudaStream_t stream);

// Exponential-unit probe: one CTA of kEx2Threads per SM, eight ex2 chains
// per thread for `iters` steps; returns ex2 results per SM clock (mean over
// SMs). Synchronises the stream.
constexpr int kEx2Threads = 512;
constexpr int kEx2MaxSms = 1024;
cudaError_t measure_ex2_rate(int num_sms, int iters, double* per_sm_per_cycle, cudaStream_t stream);

struct BwdParams {
  float* ws_lse2;                  // [BH, NQP] LSE * log2(e), +inf in the padding rows
  float* ws_d;                     // [BH, NQP] rowsum(dO * O), 0 in the padding rows
  float* ws_dq;                    // [BH, N, d] fp32 dQ accumulator (unscaled, TMA reduce-add target);
                                   // null when the workspace holds only the LSE and D parts
  unsigned* status;                // device status word
  int N, NQP;                      // query positions; NQP = N rounded up to a multiple of 128
  int Nk, NKP;                     // key positions and Nk rounded up to a multiple of 128
  int causal_off;                  // Nk - N (bottom-right causal alignment)
  int Hq, Hkv, BH, BHkv;           // BH = B*Hq, BHkv = B*Hkv
  int causal;
  float scale, scale_log2;
  unsigned long long timeout_ns;
  // optional block mask, laid out as in FwdParams; nullptr = dense. With a
  // mask, ws_count[c] and ws_list[c * G * NQP/128 ...] hold the active steps
  // (query tile | head-in-group << 16) of dK/dV CTA c = key tile * BHkv + b*Hkv + hk.
  const unsigned char* mask;
  long long mask_sb, mask_sh;
  int mask_nt;
  int* ws_count;
  unsigned* ws_list;
  int test_stall;                  // 1: the issuer first waits on a barrier nothing arrives on (timeout test)
  int head_group;                  // dK/dV: KV heads scheduled together (set by launch_bwd_dkdv)
  unsigned long long* clock_acc;   // [2] SM cycles and ns of every CTA's lifetime, summed (dK/dV); may be null
};
struct BwdMaps {
  CUtensorMap q, k, v, dO, dk, dv;
  CUtensorMap dqacc;               // fp32 [BH, N, d] accumulator, boxes of 32 columns (fa_bwd)
  CUtensorMap dq;                  // bf16 dQ output (deterministic backward)
};

// The three backward phases, each one launch on `stream`, d in {64, 128}.
cudaError_t launch_bwd_pre(int d, const void* o, const void* dO, const float* lse, const BwdParams& p, int num_sms,
                           cudaStream_t stream);
cudaError_t launch_bwd_dkdv(int d, const BwdMaps& m, const BwdParams& p, cudaStream_t stream);
// block-sparse backward: compacts each dK/dV CTA's active (head, query tile) steps
cudaError_t launch_bwd_blocklist(const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd_dq(int d, void* dq, const BwdParams& p, int num_sms, cudaStream_t stream);

// Head dims 136..256 after launch_bwd_pre (a workspace with the LSE and D
// parts only): the dV, dK and dQ passes, three launches on `stream`. m holds
// maps with 128-row boxes (q, k, v, dO, dk, dv, dq), m64 maps with 64-row
// boxes (q, dO, k, v) for the 64-row sub-tiles.
cudaError_t launch_bwd_wide(const BwdMaps& m, const BwdMaps& m64, const BwdParams& p, cudaStream_t stream);

// Deterministic backward after launch_bwd_pre: the dK/dV pass and the dQ pass
// (two launches on `stream`); reads only the LSE and D parts of the workspace.
cudaError_t launch_bwd_deterministic(int d, const BwdMaps& m, const BwdParams& p, cudaStream_t stream);

}  // namespace fa
