// FP8 (e4m3) forward on sm_103a: block-scaled quantisers and the attention
// kernel that reads their output.
//
// Method: "Flash Attention V3技术解析" section 1.3 (FP8 operands need the
// contracted dimension contiguous, so P V reads V transposed; block-wise
// quantisation) and section 3.2 (one scale per block from its largest
// magnitude); "4.3 FlashAttention-2与FlashAttention-3演进", FlashAttention-3
// section 2 (FP8 halves data movement and multiply work while the softmax
// statistics stay in higher precision). The rest of the computation is the
// bf16 forward's: tiled online softmax, output divided by the row sum once.
//
// Quantisation (e4m3, largest finite value 448): Q and K get one fp32 scale
// per block of 64 rows over all d columns, V one per column of each head over
// all keys, scale = max|block| / 448 (1 for an all-zero block), code =
// e4m3(x / scale) rounded to nearest even with saturation. A scale that
// varied along d would not factor out of Q K^T; V's per-column scales factor
// out of P V and are applied to the output columns. V is stored transposed,
// [BH, d, NP] with NP = N rounded up to 128 and zero codes past N.
//
// Attention kernel: two 128-row query tiles per CTA (producer, issuer, two
// softmax groups of four warps, ring watcher; TMEM S0 | S1 | O0 | O1) with
// kind::f8f6f4 MMAs on 16 KB tiles, and:
//   * logits = S * scale * sq(row block) * sk(key block), the key scale
//     changing at column 64 of each 128-key tile;
//   * the accumulator is rescaled only when a row max grows by more than
//     2^4 (log2 units), so P <= 2^4 relative to the running max; 2^4 P (the
//     2^4 folded into the exponent, at most 256 < 448) is rounded to e4m3
//     into one of two shared-memory P buffers per tile, the A operand of P V;
//     the row sum uses the unrounded values. A rescale waits for the previous
//     P V, so an exact running max (a rescale on most early tiles) would put
//     that wait on the softmax's path;
//   * a softmax group signals "S consumed" as soon as S_j is in its registers,
//     so S_{j+1} is computed while it works: at e4m3 rate the tensor work of a
//     key tile is shorter than the softmax, and the chain S ready -> softmax ->
//     P V -> next S would otherwise leave the tensor core idle;
//   * O column c is multiplied by V's scale of column c and divided by l.
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

constexpr int kD = 128;                  // head dimension of the kernel (a smaller d runs in it, zero-filled)
constexpr int kTile = 128 * 128;         // 128 rows x 128 e4m3 codes: one TMA box
constexpr int kQRegion = 2 * kTile;      // a query tile's region: its codes and P buffer 0, later its bf16 O
constexpr int kStages = 8;               // K / V^T ring slots
constexpr int kThreads = 384;   // softmax warps 0-7, producer 8, issuer 9, watcher 10, idle 11
// Registers move from the last warpgroup to the two softmax warpgroups
// (setmaxnreg): 256 x 184 + 128 x 120 of the 384 x 168 launched. Softmax
// warps first: the schedulers favour lower warp indices (+2% from the order,
// +1% more from the registers, bit-identical).
constexpr uint32_t kRegsSoftmax = 184, kRegsOther = 120;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther <= 384 * 168, "register split");
constexpr int kBarBytes = 512;
constexpr int kSmem = 2 * kQRegion + 2 * kTile + kStages * kTile + kBarBytes + 1024;   // + P buffers 1
static_assert(kSmem <= 227 * 1024, "shared memory budget");
constexpr float kE4m3Max = 448.0f;
constexpr int kRowBlock = 64;            // rows per Q / K scale

__device__ __forceinline__ float block_scale(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
}

}  // namespace

// ------------------------------------------------------------------ quantisers
// One CTA per (64-row block, head): the block's largest magnitude, its scale,
// then every value divided by the scale and rounded to e4m3.
__global__ void __launch_bounds__(256) fp8_quant_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                             uint8_t* __restrict__ out, float* __restrict__ scales,
                                                             int N, int d) {
  const int blk = blockIdx.x, bh = blockIdx.y;
  const int nb = (N + kRowBlock - 1) / kRowBlock;
  const int row0 = blk * kRowBlock;
  const int rows = min(kRowBlock, N - row0);
  const int chunks = rows * d / 8;                    // 16-byte chunks of eight bf16
  const uint4* src = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(bh) * N + row0) * d);
  uint2* dst = reinterpret_cast<uint2*>(out + (static_cast<size_t>(bh) * N + row0) * d);
  __shared__ float warp_max[8];
  float amax = 0.f;
  for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) amax = fmaxf(amax, warp_max[w]);
  const float s = block_scale(amax);
  if (threadIdx.x == 0) scales[static_cast<size_t>(bh) * nb + blk] = s;
  for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t q[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * h]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[2 * h + 1]));
      q[h] = pack_e4m3x2(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s)) |
             (pack_e4m3x2(__fdiv_rn(b.x, s), __fdiv_rn(b.y, s)) << 16);
    }
    dst[i] = make_uint2(q[0], q[1]);
  }
}

// V, pass 1: per-column largest magnitude of each head, as fp32 bits combined
// with an integer max (non-negative floats order like their bit patterns).
// One CTA per (128-key chunk, head), one thread per column.
__global__ void fp8_v_amax_kernel(const __nv_bfloat16* __restrict__ v, unsigned* __restrict__ amax_bits, int N,
                                  int d) {
  const int chunk = blockIdx.x, bh = blockIdx.y, c = threadIdx.x;
  if (c >= d) return;
  const int k0 = chunk * 128, k1 = min(N, k0 + 128);
  const __nv_bfloat16* src = v + static_cast<size_t>(bh) * N * d + c;
  float amax = 0.f;
  for (int k = k0; k < k1; ++k) amax = fmaxf(amax, fabsf(__bfloat162float(src[static_cast<size_t>(k) * d])));
  atomicMax(amax_bits + static_cast<size_t>(bh) * d + c, __float_as_uint(amax));
}

// V, pass 2: a 128-key chunk, 64 columns at a time, through shared memory into
// V^T rows (keys contiguous), each column with its own scale; keys past N get
// code 0. The last pass may hold fewer than 64 columns (d a multiple of 16):
// columns past d are neither read nor written. One CTA per (128-key chunk, head).
__global__ void __launch_bounds__(256) fp8_v_quant_kernel(const __nv_bfloat16* __restrict__ v,
                                                          const unsigned* __restrict__ amax_bits,
                                                          uint8_t* __restrict__ vt, int N, int NP, int d) {
  const int chunk = blockIdx.x, bh = blockIdx.y;
  const int k0 = chunk * 128;
  __shared__ __nv_bfloat16 tile[128][64];
  for (int c0 = 0; c0 < d; c0 += 64) {
    // 128 keys x 64 columns: 1024 chunks of eight bf16
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) {
      const int r = i >> 3, u = i & 7;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (k0 + r < N && c0 + 8 * u < d)
        val = *reinterpret_cast<const uint4*>(v + (static_cast<size_t>(bh) * N + k0 + r) * d + c0 + 8 * u);
      *reinterpret_cast<uint4*>(&tile[r][8 * u]) = val;
    }
    __syncthreads();
    // 64 V^T rows x 128 keys: 512 chunks of sixteen codes; lanes take consecutive columns
    for (int i = threadIdx.x; i < 512; i += blockDim.x) {
      const int c = i & 63, u = i >> 6;              // column, 16-key group
      if (c0 + c >= d) continue;
      const float s = block_scale(__uint_as_float(amax_bits[static_cast<size_t>(bh) * d + c0 + c]));
      uint32_t q[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = 16 * u + 4 * e;
        q[e] = pack_e4m3x2(__fdiv_rn(__bfloat162float(tile[k][c]), s), __fdiv_rn(__bfloat162float(tile[k + 1][c]), s)) |
               (pack_e4m3x2(__fdiv_rn(__bfloat162float(tile[k + 2][c]), s),
                            __fdiv_rn(__bfloat162float(tile[k + 3][c]), s)) << 16);
      }
      *reinterpret_cast<uint4*>(vt + (static_cast<size_t>(bh) * d + c0 + c) * NP + k0 + 16 * u) =
          make_uint4(q[0], q[1], q[2], q[3]);
    }
    __syncthreads();
  }
}

// V, pass 3: the per-column amax bits become the per-column scales, in place.
__global__ void fp8_v_scale_kernel(unsigned* __restrict__ amax_bits, int count) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < count) {
    float* out = reinterpret_cast<float*>(amax_bits);
    out[i] = block_scale(__uint_as_float(amax_bits[i]));
  }
}

// ------------------------------------------------------------------ attention
__global__ void __launch_bounds__(384, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_vt, const __grid_constant__ CUtensorMap map_o,
               const FwdParams p) {
  constexpr int kSt = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  // query region i: Q codes, then P buffer 0 of group i (later the bf16 O tile)
  const uint32_t s_q[2] = {base, base + kQRegion};
  const uint32_t s_p1[2] = {base + 2 * kQRegion, base + 2 * kQRegion + kTile};     // P buffer 1 of group i
  const uint32_t s_kv = base + 2 * kQRegion + 2 * kTile;
  const uint32_t bars = s_kv + kSt * kTile;
  auto p_buf = [&](int i, int j) { return (j & 1) ? s_p1[i] : s_q[i] + kTile; };
  auto bar_q_full = [&](int i) { return bars + 8u * i; };
  auto bar_kv_full = [&](int s) { return bars + 16u + 8u * s; };
  auto bar_kv_empty = [&](int s) { return bars + 16u + 8u * (kSt + s); };
  auto bar_s_full = [&](int i) { return bars + 16u + 16u * kSt + 8u * i; };
  auto bar_s_cons = [&](int i) { return bars + 32u + 16u * kSt + 8u * i; };
  // P-ready of tile i at step j is barrier (i, j % 2): a warp that holds S_{j+1}
  // early may write P_{j+1} before a slower warp (or the watcher) arrived for
  // step j, and that arrival must not count toward step j. No warp gets two
  // steps ahead: S_{j+2} waits for S-consumed of step j+1, i.e. for every warp
  // to be past step j, and for the watcher's step-j arrival before it.
  auto bar_p_ready = [&](int i, int j) { return bars + 48u + 16u * kSt + 16u * i + 8u * (j & 1); };
  auto bar_pv_done = [&](int i) { return bars + 80u + 16u * kSt + 8u * i; };
  auto bar_o_final = [&](int i) { return bars + 96u + 16u * kSt + 8u * i; };
  uint8_t* const gbars = gbase + (bars - base);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbars + 112 + 16 * kSt);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbars + 116 + 16 * kSt);
  const uint32_t bar_stall = bars + 120u + 16u * kSt;                     // nothing arrives (timeout test)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (query-tile pair, batch*head), heaviest causal pairs first
  const int lin = blockIdx.x;
  const int pair = p.num_pairs - 1 - lin / p.BH;
  const int bh = lin % p.BH;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bh_kv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int nq = (p.N + kBM - 1) / kBM;
  const int nk = (p.Nk + kBN - 1) / kBN;
  const int qt[2] = {2 * pair, 2 * pair + 1};
  // key tiles a query tile reaches: causal (bottom-right: key <= row + Nk - N),
  // up to the one holding key (last row + Nk - N), none if that is negative
  auto reach = [&](int t) {
    if (!p.causal) return nk;
    const int last = t * kBM + kBM - 1 + p.causal_off;
    return last < 0 ? 0 : min(nk, last / kBN + 1);
  };
  const bool has_tile[2] = {true, qt[1] < nq};
  const int nkv[2] = {reach(qt[0]), has_tile[1] ? reach(qt[1]) : 0};
  const int nmax = nkv[0] > nkv[1] ? nkv[0] : nkv[1];

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_q_full(i), 1);
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_s_cons(i), 129);                   // 128 softmax threads + the ring watcher
      mbar_init(bar_p_ready(i, 0), 129);
      mbar_init(bar_p_ready(i, 1), 129);
      mbar_init(bar_pv_done(i), 1);
      mbar_init(bar_o_final(i), 1);
    }
    for (int s = 0; s < kSt; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_stall, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    setmaxnreg_dec<kRegsOther>();
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_vt);
      for (int i = 0; i < 2; ++i) {
        if (nkv[i] == 0) continue;
        mbar_arrive_expect_tx(bar_q_full(i), kTile);
        tma_load_3d(s_q[i], &map_q, bar_q_full(i), 0, qt[i] * kBM, bh);
      }
      for (int c = 0; c < 2 * nmax; ++c) {
        const int slot = c % kSt;
        if (!mbar_wait(bar_kv_empty(slot), ((c / kSt) & 1u) ^ 1u, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_kv_full(slot), kTile);
        const uint32_t dst = s_kv + slot * kTile;
        if (c & 1)   // V^T tile: d rows x 128 keys, keys contiguous
          tma_load_3d(dst, &map_vt, bar_kv_full(slot), (c >> 1) * kBN, 0, bh_kv);
        else         // K tile: 128 keys x d
          tma_load_3d(dst, &map_k, bar_kv_full(slot), 0, (c >> 1) * kBN, bh_kv);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ tensor-core issuer
    setmaxnreg_dec<kRegsOther>();
    // Per key tile j: S_i(j+1) for each query tile as soon as its softmax has
    // read S_i(j) out of TMEM (and K_{j+1} has landed), then P_i(j) V_j as
    // soon as P_i(j) is in shared memory (and V_j has landed). Ring slots go
    // back by commits after their last reader.
    if (lane == 0) {
      const uint32_t idesc = make_idesc(0, 128, 128, 0, 0);   // e4m3 x e4m3 -> f32, both K-major
      bool ok = true;
      if (p.test_stall) ok = mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      for (int i = 0; i < 2 && ok; ++i)
        if (nkv[i] > 0) ok = mbar_wait(bar_q_full(i), 0, abort_flag, deadline);
      auto issue_qk = [&](int i, uint32_t sk) {
        const uint64_t qd = smem_desc_sw128(s_q[i], 16, 1024), kd = smem_desc_sw128(sk, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)
          mma_fp8_ss(tbase + 128u * i, desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc, kk > 0);
      };
      auto issue_pv = [&](int i, uint32_t sp, uint32_t svt, bool acc) {
        const uint64_t pd = smem_desc_sw128(sp, 16, 1024), vd = smem_desc_sw128(svt, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma_fp8_ss(tbase + 256u + 128u * i, desc_add(pd, kk * 32), desc_add(vd, kk * 32), idesc, acc || kk > 0);
      };
      if (ok && nmax > 0) {
        ok = mbar_wait(bar_kv_full(0), 0, abort_flag, deadline);     // K_0: only the issuer needs it first
        if (ok) {
          tc_fence_after();
          for (int i = 0; i < 2; ++i) {
            if (nkv[i] == 0) continue;
            issue_qk(i, s_kv);
            mma_commit(bar_s_full(i));
          }
          mma_commit(bar_kv_empty(0));
        }
      }
      for (int j = 0; j < nmax && ok; ++j) {
        const int slot_k = (2 * j + 2) % kSt, slot_v = (2 * j + 1) % kSt;
        bool any_s = false;
        for (int i = 0; i < 2 && ok; ++i) {
          if (j + 1 >= nkv[i]) continue;
          ok = mbar_wait(bar_s_cons(i), j & 1, abort_flag, deadline);   // S_i(j) read out, K_{j+1} landed
          if (!ok) break;
          tc_fence_after();
          issue_qk(i, s_kv + slot_k * kTile);
          mma_commit(bar_s_full(i));
          any_s = true;
        }
        if (!ok) break;
        if (any_s) mma_commit(bar_kv_empty(slot_k));
        for (int i = 0; i < 2 && ok; ++i) {
          if (j >= nkv[i]) continue;
          ok = mbar_wait(bar_p_ready(i, j), (j >> 1) & 1, abort_flag, deadline);  // P_i(j) written, V_j landed
          if (!ok) break;
          tc_fence_after();
          issue_pv(i, p_buf(i, j), s_kv + slot_v * kTile, j > 0);
          mma_commit(bar_pv_done(i));
          if (j + 1 == nkv[i]) mma_commit(bar_o_final(i));
        }
        if (ok) mma_commit(bar_kv_empty(slot_v));
      }
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ------------------------------------------------------------ ring watcher
    setmaxnreg_dec<kRegsOther>();
    // Folds "V_j landed" into P-ready(i, j) and "K_{j+1} landed" into
    // S-consumed(i, j). Parity waits only tell phase k from phase k-1, so it
    // observes every load in ring order (K_0 included) and arrives for a
    // phase only once the previous phase of that barrier has completed.
    if (warp == 10 && lane == 0) {
      bool ok = nmax == 0 || mbar_wait(bar_kv_full(0), 0, abort_flag, deadline);
      for (int j = 0; j < nmax && ok; ++j) {
        const int cv = 2 * j + 1;
        ok = mbar_wait(bar_kv_full(cv % kSt), (cv / kSt) & 1, abort_flag, deadline);
        for (int i = 0; i < 2 && ok; ++i) {
          if (j >= nkv[i]) continue;
          if (j >= 2) ok = mbar_wait(bar_p_ready(i, j), ((j >> 1) - 1) & 1, abort_flag, deadline);
          if (ok) mbar_arrive(bar_p_ready(i, j));
        }
        if (!ok || j + 1 >= nmax) continue;
        const int ck = 2 * j + 2;
        ok = mbar_wait(bar_kv_full(ck % kSt), (ck / kSt) & 1, abort_flag, deadline);
        for (int i = 0; i < 2 && ok; ++i) {
          if (j + 1 >= nkv[i]) continue;
          if (j > 0) ok = mbar_wait(bar_s_cons(i), (j - 1) & 1, abort_flag, deadline);
          if (ok) mbar_arrive(bar_s_cons(i));
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax groups
    setmaxnreg_inc<kRegsSoftmax>();
    const int g = warp >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int n_kv = nkv[g];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tbase + lane_off + 128u * g;
    const uint32_t t_o = tbase + lane_off + 256u + 128u * g;
    const int q_row = qt[g] * kBM + row;
    const int nqb = (p.N + kRowBlock - 1) / kRowBlock;
    const float sq = p.q_scale[static_cast<size_t>(bh) * nqb + min(q_row / kRowBlock, nqb - 1)];
    const int nkb = (p.Nk + kRowBlock - 1) / kRowBlock;
    const float* ksc = p.k_scale + static_cast<size_t>(bh_kv) * nkb;
    const float csq = p.scale_log2 * sq;
    float m = -INFINITY;                           // running max (up to 2^4 stale), log2 units
    float l = 0.f;                                 // running sum of 2^4 P
    bool ok = n_kv > 0;
    for (int j = 0; j < n_kv && ok; ++j) {
      ok = mbar_wait(bar_s_full(g), j & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld_32x32b_x32(t_s + q4 * 32, sr[q4]);
      tmem_wait_ld();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) reg_fence_x32(sr[q4]);
      if (j + 1 < n_kv) {
        // S_j is in registers: the tensor core may write S_{j+1} over it
        tc_fence_before();
        mbar_arrive(bar_s_cons(g));
      }
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      const int kv0 = j * kBN;
      int lim = kBN;
      if (p.causal) lim = min(lim, q_row + p.causal_off - kv0 + 1);
      if (kv0 + kBN > p.Nk) lim = min(lim, p.Nk - kv0);
      if (lim < kBN) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      // per-half multipliers: scale * log2(e) * sq * sk (key blocks of 64)
      const float c0 = csq * ksc[min(2 * j, nkb - 1)];
      const float c1 = csq * ksc[min(2 * j + 1, nkb - 1)];
      float mk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float* v = s + 32 * k;
        float a = fmax3(v[0], v[1], v[2]);
#pragma unroll
        for (int e = 3; e < 31; e += 2) a = fmax3(a, v[e], v[e + 1]);
        mk[k] = fmaxf(a, v[31]);
      }
      const float mx = fmaxf(fmaxf(mk[0], mk[1]) * c0, fmaxf(mk[2], mk[3]) * c1);
      const bool grow = mx > m + 4.0f;             // also true on the first tile (m = -inf)
      const float m_new = grow ? mx : m;
      const float alpha = grow ? ex2_approx(m - m_new) : 1.0f;
      m = m_new;
      // 2^4 P = 2^(s c - m + 4) <= 256; a row with no visible key yet keeps P = 0
      const float off = (m == -INFINITY) ? 0.f : 4.0f - m;
      float sum0 = 0.f, sum1 = 0.f;
      // P_j codes into shared memory buffer j % 2 (K-major, 128-byte swizzle),
      // 16 codes per store; the P V that read this buffer two tiles ago has
      // completed (it was issued before S_j)
      const uint32_t pb = p_buf(g, j);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float cm = (u < 4) ? c0 : c1;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 16 * u + 4 * e;
          float x0, x1, x2, x3;
          fma2_bc(x0, x1, s[c], s[c + 1], cm, off);
          fma2_bc(x2, x3, s[c + 2], s[c + 3], cm, off);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          add2_acc(sum0, sum1, p0, p1);
          add2_acc(sum0, sum1, p2, p3);
          w[e] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(pb, row, u)),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
      }
      l = l * alpha + (sum0 + sum1);
      // O <- alpha O before P_j V_j accumulates. P_{j-1} V_{j-1} may still be
      // running (S_j was issued before it), so wait for it: phases of that
      // barrier up to j-2 have completed and phase j cannot complete before
      // this thread's P_j, so the parity wait is unambiguous.
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        bool w = mbar_wait(bar_pv_done(g), (j - 1) & 1, abort_flag, deadline);
        w = __all_sync(0xffffffffu, w);
        if (!w) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kD; cc += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + cc, o);
          tmem_wait_ld();
          reg_fence_x32(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x32(t_o + cc, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();                    // the P codes, for the tensor core
      tc_fence_before();
      mbar_arrive(bar_p_ready(g, j));
    }
    // ---------------------------------------------------------- epilogue
    const bool empty = has_tile[g] && n_kv == 0;
    if (ok) {
      ok = mbar_wait(bar_o_final(g), 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok || empty) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      // V's scales: one per column of the head's d (columns past d hold zeros)
      const float* vsc = p.v_scale + static_cast<size_t>(bh_kv) * p.head_dim;
      auto vscale = [&](int c) { return c < p.head_dim ? __ldg(vsc + c) : 0.f; };
      // bf16 O staged over this tile's region (its Q codes and P buffer 0 are
      // no longer read: every MMA of this tile has completed)
      const uint32_t stage = s_q[g];
#pragma unroll
      for (int c0 = 0; c0 < kD; c0 += 32) {
        uint32_t o[32];
        if (!empty) {
          tmem_ld_32x32b_x32(t_o + c0, o);
          tmem_wait_ld();
          reg_fence_x32(o);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0u;
        }
        const uint32_t box = stage + (c0 / 64) * kBoxBytes;
        const int u0 = (c0 % 64) / 8;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 8 * u + 2 * e;
            w[e] = pack_bf16x2(__uint_as_float(o[c]) * (vscale(c0 + c) * inv_l),
                               __uint_as_float(o[c + 1]) * (vscale(c0 + c + 1) * inv_l));
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, row, u0 + u)),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
        }
      }
      fence_proxy_async_smem();
      // LSE = ln(sum_j e^{logit}) = (m + log2(l) - 4) ln 2, l holding 2^4 P
      if (q_row < p.N)
        p.lse[static_cast<size_t>(bh) * p.N + q_row] = l > 0.f ? (m + log2f(l) - 4.0f) * kLn2 : -INFINITY;
    }
    named_bar_sync(1 + g, 128);
    if (has_tile[g] && !*abort_flag && warp == 4 * g && lane == 0) {
      // 64-column boxes; one that would start at or past d (d <= 64) is skipped
      for (int bx = 0; bx < 2; ++bx)
        if (bx * 64 < p.head_dim) tma_store_3d(&map_o, s_q[g] + bx * kBoxBytes, bx * 64, qt[g] * kBM, bh);
      tma_store_commit();
      tma_store_wait_all0();
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) atomicOr(p.status, kDevTimeout);
    abort_grace_period();
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

cudaError_t launch_fp8_quant_rows(const void* x, void* out, float* scales, int BH, int N, int d,
                                  cudaStream_t stream) {
  const dim3 grid((N + kRowBlock - 1) / kRowBlock, BH);
  fp8_quant_rows_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), static_cast<uint8_t*>(out),
                                                  scales, N, d);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quant_v(const void* v, void* vt, float* scales, int BH, int N, int d, cudaStream_t stream) {
  const int NP = (N + 127) / 128 * 128;
  cudaError_t e = cudaMemsetAsync(scales, 0, static_cast<size_t>(BH) * d * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const dim3 grid(NP / 128, BH);
  unsigned* bits = reinterpret_cast<unsigned*>(scales);
  fp8_v_amax_kernel<<<grid, d, 0, stream>>>(static_cast<const __nv_bfloat16*>(v), bits, N, d);
  fp8_v_quant_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(v), bits, static_cast<uint8_t*>(vt),
                                               N, NP, d);
  const int count = BH * d;
  fp8_v_scale_kernel<<<(count + 255) / 256, 256, 0, stream>>>(bits, count);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mvt,
                           const CUtensorMap& mo, FwdParams p, cudaStream_t stream) {
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    return cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e != cudaSuccess) return e;
  const int nq = (p.N + kBM - 1) / kBM;
  p.num_pairs = (nq + 1) / 2;
  fwd_fp8_kernel<<<p.num_pairs * p.BH, kThreads, kSmem, stream>>>(mq, mk, mvt, mo, p);
  return cudaGetLastError();
}

}  // namespace fa
