// Deterministic backward on sm_103a: dQ, dK, dV of <O, dO> with every output
// bit reproducible from run to run.
//
// The default backward (fa_bwd.cu) adds each key tile's dQ contribution into
// an fp32 accumulator with TMA reduce-add, so the order of the additions, and
// with it the last bits of dQ, depends on scheduling. Here dQ is computed in a
// pass of its own that recomputes the scores ("Flash Attention V3技术解析"
// 2.1 "梯度计算" describes the atomic accumulation this replaces): one CTA per
// query tile walks the key tiles it sees and keeps dQ in TMEM, so every dQ
// element is a fixed sequence of additions. It costs two more GEMMs per tile
// pair (S and dP are formed twice), about 40% more tensor work than fa_bwd.
//
//  det_dkdv_kernel   one CTA per 128-key tile of one (batch, KV head); for
//                    each query head of the group and each query tile that
//                    sees these keys:
//                      S^T = K Q_i^T, dP^T = V dO_i^T          (TMEM)
//                      P^T = 2^(S^T s log2e - LSE_i log2e)      (over S^T, bf16)
//                      dS^T = P^T (dP^T - D_i)                  (over dP^T, bf16)
//                      dV += P^T dO_i, dK += dS^T Q_i          (A from TMEM)
//                    then dK *= scale; dK, dV stored once.
//  det_dq_kernel     one CTA per 128-row query tile; for each key tile it
//                    sees: S = Q K_j^T, dP = dO V_j^T, dS = P (dP - D) (over S,
//                    bf16), dQ += dS K_j (A from TMEM); dQ *= scale, stored once.
// Both read D and the base-2 LSE that bwd_pre_kernel (fa_bwd.cu) writes.
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

// Shared pieces of the two tensor-core kernels.
template <int D>
struct DetTile {
  static constexpr int kNBox = D / 64;                  // bf16: 64 elements per 128-byte row
  static constexpr int kTileBytes = kNBox * kBoxBytes;  // one [128, D] bf16 tile
};

// Stage the fp32 TMEM columns [0, D/2) at `taddr` (this thread's lane), times
// `mul`, as bf16 columns [c_begin, c_begin + D/2) of a [128, D]
// 128-byte-swizzled tile at `stg`.
template <int D>
__device__ __forceinline__ void stage_half_bf16(uint32_t taddr, uint32_t stg, int row, int c_begin, float mul) {
#pragma unroll
  for (int c0 = 0; c0 < D / 2; c0 += 32) {
    uint32_t t[32];
    tmem_ld_32x32b_x32(taddr + c0, t);
    tmem_wait_ld();
    reg_fence_x32(t);
    const int col = c_begin + c0;
    const uint32_t box = stg + (col / 64) * kBoxBytes;
    const int u0 = (col % 64) / 8;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = pack_bf16x2(__uint_as_float(t[8 * u + 2 * e]) * mul, __uint_as_float(t[8 * u + 2 * e + 1]) * mul);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, row, u0 + u)),
                   "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
    }
  }
}

// ------------------------------------------------------------------ dK / dV
template <int D>
struct DetDkdvCfg : DetTile<D> {
  using DetTile<D>::kTileBytes;
  static constexpr int kVecBytes = 512;                // 128 fp32 (LSE or D of one query tile)
  // shared memory: K | V | stage0 {Q, dO} | stage1 {Q, dO} | lse2[2] | D[2] | barriers
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffStage = 2 * kTileBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffVec = kOffStage + 2 * kStageBytes;
  static constexpr int kOffBar = kOffVec + 4 * kVecBytes;
  static constexpr int kSmemBytes = kOffBar + 128 + 1024;   // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
  static constexpr int kThreads = 320;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(2 * D + 256 <= 512, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(320, 1)
det_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
                const BwdParams p) {
  using C = DetDkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t s_k = base + C::kOffK, s_v = base + C::kOffV;
  auto s_q = [&](int st) { return base + C::kOffStage + st * C::kStageBytes; };
  auto s_do = [&](int st) { return base + C::kOffStage + st * C::kStageBytes + C::kTileBytes; };
  auto s_lse = [&](int st) { return base + C::kOffVec + st * C::kVecBytes; };
  auto s_dvec = [&](int st) { return base + C::kOffVec + (2 + st) * C::kVecBytes; };
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_kv_full = bars;
  auto bar_q_full = [&](int st) { return bars + 8u + 8u * st; };
  auto bar_q_empty = [&](int st) { return bars + 24u + 8u * st; };
  const uint32_t bar_s_full = bars + 40, bar_dp_full = bars + 48, bar_p_ready = bars + 56;
  const uint32_t bar_ds_ready = bars + 64, bar_o_final = bars + 72;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 80);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 84);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (key tile, batch * kv head); the key tiles with the most
  // query tiles to visit (small index when causal) go first
  const int jt = blockIdx.x / p.BHkv;
  const int bhkv = blockIdx.x % p.BHkv;
  const int b = bhkv / p.Hkv, hk = bhkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int nq = p.NQP / kBM;
  const int it0 = p.causal ? jt : 0;
  const int tiles_per_head = nq - it0;
  const int nsteps = G * tiles_per_head;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_kv_full, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(bar_q_full(st), 1);
      mbar_init(bar_q_empty(st), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_p_ready, 256);
    mbar_init(bar_ds_ready, 256);
    mbar_init(bar_o_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_do);
      mbar_arrive_expect_tx(bar_kv_full, 2 * C::kTileBytes);
      for (int bx = 0; bx < C::kNBox; ++bx) {
        tma_load_3d(s_k + bx * kBoxBytes, &map_k, bar_kv_full, bx * 64, jt * kBN, bhkv);
        tma_load_3d(s_v + bx * kBoxBytes, &map_v, bar_kv_full, bx * 64, jt * kBN, bhkv);
      }
      for (int step = 0; step < nsteps; ++step) {
        const int st = step & 1;
        if (!mbar_wait(bar_q_empty(st), ((step >> 1) & 1) ^ 1, abort_flag, deadline)) break;
        const int h = hk * G + step / tiles_per_head;
        const int it = it0 + step % tiles_per_head;
        const int bh = b * p.Hq + h;
        mbar_arrive_expect_tx(bar_q_full(st), 2 * C::kTileBytes + 2 * C::kVecBytes);
        for (int bx = 0; bx < C::kNBox; ++bx) {
          tma_load_3d(s_q(st) + bx * kBoxBytes, &map_q, bar_q_full(st), bx * 64, it * kBM, bh);
          tma_load_3d(s_do(st) + bx * kBoxBytes, &map_do, bar_q_full(st), bx * 64, it * kBM, bh);
        }
        const size_t voff = static_cast<size_t>(bh) * p.NQP + static_cast<size_t>(it) * kBM;
        bulk_load(s_lse(st), p.ws_lse2 + voff, C::kVecBytes, bar_q_full(st));
        bulk_load(s_dvec(st), p.ws_d + voff, C::kVecBytes, bar_q_full(st));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ tensor-core issuer
    // Issue order S_0 | dP_0, [P_0] dV_0, S_1, [dS_0] dK_0 | dP_1, [P_1] dV_1,
    // S_2, [dS_1] dK_1 | ...: the next tile's S^T goes in as soon as dV has
    // consumed P^T (it overwrites those columns), so the softmax groups' P
    // phase of tile i+1 overlaps dK_i and dP_{i+1}. dP^T overwrites the dS^T
    // columns after dK, its reader; the tensor core runs one thread's MMAs in
    // issue order.
    if (lane == 0) {
      const uint32_t id_kk = make_idesc(1, 128, 128, 0, 0);  // S^T, dP^T: both operands K-major
      const uint32_t id_tmn = make_idesc(1, 128, D, 0, 1);   // dV, dK: A from TMEM, B MN-major
      const uint64_t k_kmaj = smem_desc_sw128(s_k, 16, 1024), v_kmaj = smem_desc_sw128(s_v, 16, 1024);
      const uint64_t q_kmaj[2] = {smem_desc_sw128(s_q(0), 16, 1024), smem_desc_sw128(s_q(1), 16, 1024)};
      const uint64_t q_mn[2] = {smem_desc_sw128(s_q(0), kBoxBytes, 1024), smem_desc_sw128(s_q(1), kBoxBytes, 1024)};
      const uint64_t do_kmaj[2] = {smem_desc_sw128(s_do(0), 16, 1024), smem_desc_sw128(s_do(1), 16, 1024)};
      const uint64_t do_mn[2] = {smem_desc_sw128(s_do(0), kBoxBytes, 1024), smem_desc_sw128(s_do(1), kBoxBytes, 1024)};
      auto issue_s = [&](int st) {                         // S^T = K Q^T
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColS, desc_add(k_kmaj, off), desc_add(st ? q_kmaj[1] : q_kmaj[0], off), id_kk,
                      kk > 0);
        }
        mma_commit(bar_s_full);
      };
      bool ok = mbar_wait(bar_kv_full, 0, abort_flag, deadline) && mbar_wait(bar_q_full(0), 0, abort_flag, deadline);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int step = 0; step < nsteps && ok; ++step) {
        const int st = step & 1;
        const uint64_t qm = st ? q_mn[1] : q_mn[0];
        const uint64_t dok = st ? do_kmaj[1] : do_kmaj[0], dom = st ? do_mn[1] : do_mn[0];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {                // dP^T = V dO^T
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColDP, desc_add(v_kmaj, off), desc_add(dok, off), id_kk, kk > 0);
        }
        mma_commit(bar_dp_full);
        if (!mbar_wait(bar_p_ready, step & 1, abort_flag, deadline)) { ok = false; break; }
        tc_fence_after();
        // dV += P^T dO  (K = 128 queries; P^T of query q sits in S column 64*(q/64) + (q%64)/2)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tbase + C::kColDV, tbase + C::kColS + 64 * (kk >> 2) + (kk & 3) * 8,
                      desc_add(dom, kk * 16 * 128), id_tmn, step > 0 || kk > 0);
        if (step + 1 < nsteps) {
          if (!mbar_wait(bar_q_full(st ^ 1), ((step + 1) >> 1) & 1, abort_flag, deadline)) { ok = false; break; }
          tc_fence_after();
          issue_s(st ^ 1);
        }
        if (!mbar_wait(bar_ds_ready, step & 1, abort_flag, deadline)) { ok = false; break; }
        tc_fence_after();
        // dK += dS^T Q  (dS^T of query q sits in dP column 64*(q/64) + (q%64)/2)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tbase + C::kColDK, tbase + C::kColDP + 64 * (kk >> 2) + (kk & 3) * 8,
                      desc_add(qm, kk * 16 * 128), id_tmn, step > 0 || kk > 0);
        mma_commit(bar_q_empty(st));       // Q, dO, LSE, D of this step are no longer read
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax-gradient groups
    const int g = (warp - 2) >> 2;                 // query-column half: [64g, 64g + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // key row (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool key_pad = jt * kBN + r >= p.N;      // key rows past N contribute nothing
    bool ok = true;
    for (int step = 0; step < nsteps && ok; ++step) {
      const int st = step & 1;
      const int it = it0 + step % tiles_per_head;
      const bool diag = p.causal && it == jt;
      ok = mbar_wait(bar_q_full(st), (step >> 1) & 1, abort_flag, deadline) &&
           mbar_wait(bar_s_full, step & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(gbase + (s_lse(st) - base));
      const float* dvec = reinterpret_cast<const float*>(gbase + (s_dvec(st) - base));
      // ---- phase A (overlaps the dP^T MMA): P^T = 2^(S^T s log2e - LSE log2e),
      // written over the S^T columns this group has read, as bf16 pairs
      float pf[64];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * g + 32 * ch;            // first query column of this chunk
        uint32_t sv[32];
        tmem_ld_32x32b_x32(tbase + lane_off + C::kColS + c0, sv);
        tmem_wait_ld();
        reg_fence_x32(sv);
        const float4* l4 = reinterpret_cast<const float4*>(lse2 + c0);
        uint32_t pp[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 lv = l4[c / 4];
          const float lq[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv = ex2_approx(fmaf(__uint_as_float(sv[c + e]), sl2, -lq[e]));
            if (key_pad || (diag && c0 + c + e < r)) pv = 0.f;
            pf[32 * ch + c + e] = pv;
          }
          pp[c / 2] = pack_bf16x2(pf[32 * ch + c], pf[32 * ch + c + 1]);
          pp[c / 2 + 1] = pack_bf16x2(pf[32 * ch + c + 2], pf[32 * ch + c + 3]);
        }
        tmem_st_32x32b_x16(tbase + lane_off + C::kColS + 64 * g + 16 * ch, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p_ready);
      // ---- phase B (overlaps the dV MMA): dS^T = P^T (dP^T - D), written over
      // the dP^T columns this group has read, as bf16 pairs
      ok = mbar_wait(bar_dp_full, step & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = 64 * g + 32 * ch;
        uint32_t dp[32];
        tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + c0, dp);
        tmem_wait_ld();
        reg_fence_x32(dp);
        const float4* d4 = reinterpret_cast<const float4*>(dvec + c0);
        uint32_t dd[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 dv4 = d4[c / 4];
          const float dq4[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
          float ds[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) ds[e] = pf[32 * ch + c + e] * (__uint_as_float(dp[c + e]) - dq4[e]);
          dd[c / 2] = pack_bf16x2(ds[0], ds[1]);
          dd[c / 2 + 1] = pack_bf16x2(ds[2], ds[3]);
        }
        tmem_st_32x32b_x16(tbase + lane_off + C::kColDP + 64 * g + 16 * ch, dd);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ds_ready);
    }
    // ---------------------------------------------------------- dK, dV epilogue
    if (ok) {
      ok = mbar_wait(bar_o_final, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      // staging: the V buffer for dV and the K buffer for dK (every MMA has completed)
      stage_half_bf16<D>(tbase + lane_off + C::kColDV + g * (D / 2), s_v, r, g * (D / 2), 1.0f);
      stage_half_bf16<D>(tbase + lane_off + C::kColDK + g * (D / 2), s_k, r, g * (D / 2), p.scale);
      fence_proxy_async_smem();
    }
    // all eight warps meet here whether or not their waits succeeded; a warp
    // that gave up has raised the abort flag: store nothing
    named_bar_sync(1, 256);
    if (!*abort_flag && warp == 2 && lane == 0) {
      for (int bx = 0; bx < C::kNBox; ++bx) {
        tma_store_3d(&map_dv, s_v + bx * kBoxBytes, bx * 64, jt * kBN, bhkv);
        tma_store_3d(&map_dk, s_k + bx * kBoxBytes, bx * 64, jt * kBN, bhkv);
      }
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
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

// ------------------------------------------------------------------ dQ
template <int D>
struct DetDqCfg : DetTile<D> {
  using DetTile<D>::kTileBytes;
  // K/V slot ring. A K tile stays in use from S_j until dQ_j completes, so
  // the ring needs room for the producer to run ahead of that.
  static constexpr int kStages = 5;
  // shared memory: Q | dO | ring[kStages] | barriers
  static constexpr int kOffQ = 0;
  static constexpr int kOffDo = kTileBytes;
  static constexpr int kOffRing = 2 * kTileBytes;
  static constexpr int kOffBar = kOffRing + kStages * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // S is double-buffered: S_j in buffer j&1 while the tensor core already
  // computes S_{j+1} into the other
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColDP = 256, kColDQ = 384;
  static constexpr int kThreads = 320;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(384 + D <= 512, "TMEM budget");
};

template <int D>
__global__ void __launch_bounds__(320, 1)
det_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
              const __grid_constant__ CUtensorMap map_dq, const BwdParams p) {
  using C = DetDqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t s_q = base + C::kOffQ, s_do = base + C::kOffDo, s_ring = base + C::kOffRing;
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_q_full = bars;
  auto bar_kv_full = [&](int s) { return bars + 8u + 8u * s; };                    // kStages
  auto bar_kv_empty = [&](int s) { return bars + 8u + 8u * (C::kStages + s); };    // kStages
  auto bar_s_full = [&](int x) { return bars + 8u + 16u * C::kStages + 8u * x; };  // 2
  const uint32_t bar_dp_full = bars + 24 + 16 * C::kStages;
  const uint32_t bar_dp_read = bars + 32 + 16 * C::kStages;
  // dS-ready of key tile j is barrier j % 2. A warp that has written dS_j may
  // already hold S_{j+1} (issued before the dP-read wait) and dP_{j+1} (issued
  // once every warp has read dP_j) and arrive for tile j+1 while a slower warp
  // is still writing dS_j: with one barrier that arrival would complete tile
  // j's phase early. No warp gets two tiles ahead: dP_{j+2} waits for every
  // warp to read dP_{j+1}, which each does after its tile-j arrival.
  auto bar_ds_ready = [&](int j) { return bars + 40u + 16u * C::kStages + 8u * (j & 1); };
  const uint32_t bar_dq_final = bars + 56 + 16 * C::kStages;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 64 + 16 * C::kStages);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 68 + 16 * C::kStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (query tile, batch * head); the longest causal rows first
  const int nq = p.NQP / kBM;
  const int it = nq - 1 - static_cast<int>(blockIdx.x / p.BH);
  const int bh = blockIdx.x % p.BH;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bhkv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int n_kv = p.causal ? it + 1 : nq;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_s_full(0), 1);
    mbar_init(bar_s_full(1), 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_dp_read, 256);
    mbar_init(bar_ds_ready(0), 256);
    mbar_init(bar_ds_ready(1), 256);
    mbar_init(bar_dq_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      mbar_arrive_expect_tx(bar_q_full, 2 * C::kTileBytes);
      for (int bx = 0; bx < C::kNBox; ++bx) {
        tma_load_3d(s_q + bx * kBoxBytes, &map_q, bar_q_full, bx * 64, it * kBM, bh);
        tma_load_3d(s_do + bx * kBoxBytes, &map_do, bar_q_full, bx * 64, it * kBM, bh);
      }
      for (int c = 0; c < 2 * n_kv; ++c) {             // K_0, V_0, K_1, V_1, ...
        const int slot = c % C::kStages;
        if (!mbar_wait(bar_kv_empty(slot), ((c / C::kStages) & 1) ^ 1, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_kv_full(slot), C::kTileBytes);
        const CUtensorMap* m = (c & 1) ? &map_v : &map_k;
        const uint32_t dst = s_ring + slot * C::kTileBytes;
        for (int bx = 0; bx < C::kNBox; ++bx)
          tma_load_3d(dst + bx * kBoxBytes, m, bar_kv_full(slot), bx * 64, (c >> 1) * kBN, bhkv);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ tensor-core issuer
    // S_0, dP_0; then per key tile j: S_{j+1} (other S buffer), [dP_j read]
    // dP_{j+1}, [dS_j ready] dQ += dS_j K_j. K_j is released after dQ_j, V_j
    // after dP_j. With 5 slots a slot alternates K and V tiles; the tile
    // loaded into a slot is always released after the one loaded before it
    // (K_j before V_{j+2}, V_j before K_{j+3}), so each slot's releases stay
    // in its load order.
    if (lane == 0) {
      const uint32_t id_kk = make_idesc(1, 128, 128, 0, 0);  // S, dP: both operands K-major
      const uint32_t id_tmn = make_idesc(1, 128, D, 0, 1);   // dQ: A = dS from TMEM, B = K MN-major
      const uint64_t q_kmaj = smem_desc_sw128(s_q, 16, 1024), do_kmaj = smem_desc_sw128(s_do, 16, 1024);
      int c = 0;
      auto take = [&](int& slot) -> bool {
        slot = c % C::kStages;
        const bool r = mbar_wait(bar_kv_full(slot), (c / C::kStages) & 1, abort_flag, deadline);
        ++c;
        return r;
      };
      auto slot_kmaj = [&](int slot) { return smem_desc_sw128(s_ring + slot * C::kTileBytes, 16, 1024); };
      auto slot_mn = [&](int slot) { return smem_desc_sw128(s_ring + slot * C::kTileBytes, kBoxBytes, 1024); };
      auto issue_s = [&](uint32_t col, uint64_t kd) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + col, desc_add(q_kmaj, off), desc_add(kd, off), id_kk, kk > 0);
        }
      };
      auto issue_dp = [&](uint64_t vd) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColDP, desc_add(do_kmaj, off), desc_add(vd, off), id_kk, kk > 0);
        }
      };
      bool ok = mbar_wait(bar_q_full, 0, abort_flag, deadline);
      int kslot = 0, vslot = 0;
      if (ok) ok = take(kslot);
      if (ok) {
        tc_fence_after();
        issue_s(C::kColS0, slot_kmaj(kslot));
        mma_commit(bar_s_full(0));
        ok = take(vslot);
      }
      if (ok) {
        tc_fence_after();
        issue_dp(slot_kmaj(vslot));
        mma_commit(bar_dp_full);
        mma_commit(bar_kv_empty(vslot));
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int x = j & 1;
        const int kslot_j = kslot;
        if (j + 1 < n_kv) {
          if (!take(kslot)) { ok = false; break; }
          tc_fence_after();
          issue_s(x ? C::kColS0 : C::kColS1, slot_kmaj(kslot));
          mma_commit(bar_s_full(x ^ 1));
        }
        if (!mbar_wait(bar_dp_read, j & 1, abort_flag, deadline)) { ok = false; break; }
        if (j + 1 < n_kv) {
          if (!take(vslot)) { ok = false; break; }
          tc_fence_after();
          issue_dp(slot_kmaj(vslot));
          mma_commit(bar_dp_full);
          mma_commit(bar_kv_empty(vslot));
        }
        if (!mbar_wait(bar_ds_ready(j), (j >> 1) & 1, abort_flag, deadline)) { ok = false; break; }
        tc_fence_after();
        // dQ += dS_j K_j  (K = 128 keys; dS of key k sits in column S_x + 64*(k/64) + (k%64)/2)
        const uint64_t km = slot_mn(kslot_j);
        const uint32_t scol = x ? C::kColS1 : C::kColS0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tbase + C::kColDQ, tbase + scol + 64 * (kk >> 2) + (kk & 3) * 8, desc_add(km, kk * 16 * 128),
                      id_tmn, j > 0 || kk > 0);
        mma_commit(bar_kv_empty(kslot_j));
      }
      if (ok) mma_commit(bar_dq_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax-gradient groups
    const int g = (warp - 2) >> 2;                 // key-column half: [64g, 64g + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // query row within the tile (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const size_t vrow = static_cast<size_t>(bh) * p.NQP + static_cast<size_t>(it) * kBM + r;
    const float lse2 = p.ws_lse2[vrow];            // +inf on padded rows: P = 0 there
    const float drow = p.ws_d[vrow];
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int x = j & 1;
      const uint32_t scol = x ? C::kColS1 : C::kColS0;
      ok = mbar_wait(bar_s_full(x), (j >> 1) & 1, abort_flag, deadline) &&
           mbar_wait(bar_dp_full, j & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[2][32], dp[2][32];
      tmem_ld_32x32b_x32(tbase + lane_off + scol + 64 * g, sv[0]);
      tmem_ld_32x32b_x32(tbase + lane_off + scol + 64 * g + 32, sv[1]);
      tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + 64 * g, dp[0]);
      tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + 64 * g + 32, dp[1]);
      tmem_wait_ld();
      reg_fence_x32(sv[0]);
      reg_fence_x32(sv[1]);
      reg_fence_x32(dp[0]);
      reg_fence_x32(dp[1]);
      tc_fence_before();
      mbar_arrive(bar_dp_read);                    // the dP columns may be overwritten now
      // mask: keys past the diagonal (causal) and past N
      const int kv0 = j * kBN;
      int lim = kBN;
      if (p.causal && j == it) lim = r + 1;
      if (kv0 + kBN > p.N) lim = min(lim, p.N - kv0);
      uint32_t dd[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        float ds[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cc = c + e;
          float pv = ex2_approx(fmaf(__uint_as_float(sv[cc >> 5][cc & 31]), sl2, -lse2));
          if (64 * g + cc >= lim) pv = 0.f;
          ds[e] = pv * (__uint_as_float(dp[cc >> 5][cc & 31]) - drow);
        }
        dd[c / 2] = pack_bf16x2(ds[0], ds[1]);
      }
      // dS (bf16 pairs) over the S columns this group has read:
      // key k at column 64*(k/64) + (k%64)/2
      tmem_st_32x32b_x32(tbase + lane_off + scol + 64 * g, dd);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ds_ready(j));
    }
    // ---------------------------------------------------------- dQ epilogue
    if (ok) {
      ok = mbar_wait(bar_dq_final, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      // staging in the Q buffer (every MMA has completed)
      stage_half_bf16<D>(tbase + lane_off + C::kColDQ + g * (D / 2), s_q, r, g * (D / 2), p.scale);
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (!*abort_flag && warp == 2 && lane == 0) {
      for (int bx = 0; bx < C::kNBox; ++bx) tma_store_3d(&map_dq, s_q + bx * kBoxBytes, bx * 64, it * kBM, bh);
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
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

// ------------------------------------------------------------------ launch
template <int D>
static cudaError_t launch_det_d(const BwdMaps& m, const BwdParams& p, cudaStream_t stream) {
  static PerDeviceOnce attr_a, attr_b;
  cudaError_t e = attr_a.run([] {
    return cudaFuncSetAttribute(det_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                DetDkdvCfg<D>::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  e = attr_b.run([] {
    return cudaFuncSetAttribute(det_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DetDqCfg<D>::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  det_dkdv_kernel<D><<<(p.NQP / kBN) * p.BHkv, DetDkdvCfg<D>::kThreads, DetDkdvCfg<D>::kSmemBytes, stream>>>(
      m.q, m.k, m.v, m.dO, m.dk, m.dv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  det_dq_kernel<D><<<(p.NQP / kBM) * p.BH, DetDqCfg<D>::kThreads, DetDqCfg<D>::kSmemBytes, stream>>>(
      m.q, m.k, m.v, m.dO, m.dq, p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_deterministic(int d, const BwdMaps& m, const BwdParams& p, cudaStream_t stream) {
  // d < 128 runs in the kernel for the next size up: the tensor maps carry
  // the true d, so the columns past it load as zeros (adding nothing to S,
  // dP, dQ, dK or dV) and are skipped by the stores
  if (d > 64 && d <= 128) return launch_det_d<128>(m, p, stream);
  if (d >= 8 && d <= 64) return launch_det_d<64>(m, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
