// Backward exact attention on sm_103a for head dimensions 136..256 (built for
// d = 256; a smaller d reads zeros past its columns and stores none of them).
//
// Method: as fa_bwd.cu, the probabilities are recomputed from the stored
// logsumexp ("4.3 FlashAttention-2与FlashAttention-3演进", FlashAttention-3
// section 3) tile by tile (deepschool.ru FlashAttention-2, "Улучшение backward
// pass"); FlashAttention-2 extends the supported head dimension to 256 (same
// page, "Снижение накладных расходов").
//
// At d = 256 the dK and dV accumulators of a 128-key tile alone fill the 512
// TMEM columns, and one step's Q, dO, K and V tiles (64 KB each) exceed shared
// memory. The gradients are therefore formed in three passes over 128-row
// steps, each with a fixed order of additions (no atomics: every output is
// bit reproducible):
//   wide_dv_kernel  per 128-key tile: S^T = K Q_t^T, P^T -> TMEM (bf16),
//                   dV += P^T dO_t                              over query tiles t
//   wide_dk_kernel  per 128-key tile: S^T, then dP^T = V dO_t^T in the same
//                   TMEM columns, dS^T = P^T (dP^T - D) -> shared memory,
//                   dK += dS^T Q_t                              over query tiles t
//   wide_dq_kernel  per 128-row query tile: S = Q K_j^T, then dP = dO V_j^T,
//                   dS -> shared memory, dQ += dS K_j           over key tiles j
// Every score product is M = 128, N = 128, K = 256. S (or S^T) and dP are
// formed twice or three times: 8 GEMMs of the 5 the method needs.
// bwd_pre_kernel (fa_bwd.cu) writes D and the base-2 LSE first. The dK and dQ
// passes keep K or Q in TMEM as the A operand of the scores.
//
// Roles (320 threads): warps 0-7 two per TMEM lane quarter, each thread one
// lane (key row in the dV and dK passes, query row in the dQ pass) and one
// half of the step's 128 score columns (warps 0-3 the first, 4-7 the second);
// warp 8 TMA producer, warp 9 MMA issuer (one thread); warp 1 owns TMEM.
#include <algorithm>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kWD = 256;                          // head-dimension build
constexpr int kWTile = kWD / 64 * kBoxBytes;      // [128, 256] bf16: 64 KB
constexpr int kWThreads = 320;
constexpr int kWProd = 8, kWIss = 9;           // producer and issuer warps
constexpr uint32_t kWColAcc = 0;                  // TMEM: the dK, dV or dQ accumulator in columns 0-255

// 64 fp32 TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t r[2][32];
  tmem_ld_32x32b_x32(taddr, r[0]);
  tmem_ld_32x32b_x32(taddr + 32, r[1]);
  tmem_wait_ld();
  reg_fence_x32(r[0]);
  reg_fence_x32(r[1]);
#pragma unroll
  for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(r[c >> 5][c & 31]);
}

// 64 bf16 values as row `row` of a [128, 64] 128-byte-swizzled box
__device__ __forceinline__ void store_row64(uint32_t box, int row, const float (&x)[64]) {
#pragma unroll
  for (int u = 0; u < 8; ++u)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, row, u)),
                 "r"(pack_bf16x2(x[8 * u], x[8 * u + 1])), "r"(pack_bf16x2(x[8 * u + 2], x[8 * u + 3])),
                 "r"(pack_bf16x2(x[8 * u + 4], x[8 * u + 5])), "r"(pack_bf16x2(x[8 * u + 6], x[8 * u + 7]))
                 : "memory");
}

// Accumulator columns [128 half, 128 half + 128) of this thread's lane, times
// `mul`, into row `row` of a [128, 256] bf16 tile (four 128-row boxes) at `stg`
__device__ __forceinline__ void stage_acc_row(uint32_t taddr, uint32_t stg, int row, float mul, int half) {
#pragma unroll
  for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 32) {
    uint32_t t[32];
    tmem_ld_32x32b_x32(taddr + c0, t);
    tmem_wait_ld();
    reg_fence_x32(t);
    const uint32_t box = stg + (c0 / 64) * kBoxBytes;
    const int u0 = (c0 % 64) / 8;
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

}  // namespace

// ------------------------------------------------------------------ dK per key tile, 128-query steps
// Shared memory: V | two 64 KB slots | dS^T | LSE, D x2 | barriers. K lands in
// slot 0 and the warps copy it into TMEM as the A operand of S^T; Q_t then
// always goes to slot 0 and dO_t to slot 1, so dO_{t+1} loads as soon as
// dP^T_t has read dO_t, early in step t, and Q_{t+1} once dK_t has read Q_t.
// TMEM: dK accumulator | dP^T, then S^T, of the step (128 columns) | K.
// Per step dP^T_t (N = 128 queries) goes into the score columns; once every
// warp has read it into registers, S^T_t goes into the same columns; once
// every warp has written dS^T_t, dK += dS^T_t Q_t, and dP^T_{t+1} follows.
struct WideDkCfg {
  static constexpr int kOffV = 0;
  static constexpr int kOffSlot = kWTile;              // two 64 KB slots; slot 0 first holds K
  static constexpr int kOffDs = kOffSlot + 2 * kWTile;  // dS^T [128 keys, 128 queries] bf16: two boxes
  static constexpr int kOffVec = kOffDs + 2 * kBoxBytes;
  static constexpr int kVecBytes = 1024;               // LSE log2(e) and D of 128 queries
  static constexpr int kOffBar = kOffVec + 2 * kVecBytes;
  static constexpr uint32_t kColSP = 256, kColK = 384;
  static constexpr int kLayout = kOffBar + 144;
  // the per-block maximum: the layout needs the dynamic window to start within
  // 880 bytes of a 1 KB boundary (checked at run time)
  static constexpr int kSmemAlloc = 232448;
  static_assert(kLayout <= kSmemAlloc, "shared memory budget");
};

__global__ void __launch_bounds__(kWThreads, 1)
wide_dk_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
               const __grid_constant__ CUtensorMap map_dk, const BwdParams p) {
  using C = WideDkCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  if ((base - raw) + C::kLayout > static_cast<uint32_t>(C::kSmemAlloc)) {
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  const uint32_t s_v = base + C::kOffV;
  auto s_slot = [&](int i) { return base + C::kOffSlot + i * kWTile; };
  const uint32_t s_k = s_slot(0);                      // the K tile until it is in TMEM
  const uint32_t s_ds = base + C::kOffDs;
  auto s_vec = [&](int i) { return base + C::kOffVec + i * C::kVecBytes; };
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_kv_full = bars;                   // K and V landed
  auto bar_full = [&](int i) { return bars + 8u + 8u * i; };
  auto bar_empty = [&](int i) { return bars + 24u + 8u * i; };
  auto bar_vec_full = [&](int i) { return bars + 40u + 8u * i; };
  auto bar_vec_empty = [&](int i) { return bars + 56u + 8u * i; };
  const uint32_t bar_s_full = bars + 72, bar_s_read = bars + 80, bar_dp_full = bars + 88;
  const uint32_t bar_ready = bars + 96, bar_o_final = bars + 104, bar_stall = bars + 112;
  const uint32_t bar_k_tmem = bars + 120;              // every row of K copied into TMEM
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 128);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 132);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (key tile, batch * kv head); causal: small key tiles first.
  // KV heads go in groups of p.head_group whose Q and dO fit in part of L2.
  const int nkt = p.NKP / kBN;
  const int grp = blockIdx.x / (nkt * p.head_group);
  const int gsize = min(p.head_group, p.BHkv - grp * p.head_group);
  const int local = blockIdx.x - grp * p.head_group * nkt;
  const int jt = local / gsize;
  const int bhkv = grp * p.head_group + local % gsize;
  const int b = bhkv / p.Hkv, hk = bhkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int nq = p.NQP / kBM;
  // first query tile that sees key tile jt (bottom-right causal)
  const int first_row = jt * kBN - p.causal_off;
  const int it0 = p.causal ? (first_row <= 0 ? 0 : min(nq, first_row / kBM)) : 0;
  const int per_head = nq - it0;
  const int nsteps = G * per_head;
  auto step_head = [&](int t) { return b * p.Hq + hk * G + t / per_head; };
  auto step_tile = [&](int t) { return it0 + t % per_head; };
  // Q_t always in slot 0 (after K has gone from it into TMEM), dO_t in slot 1:
  // dO_{t+1} loads as soon as dP^T_t has read dO_t, early in step t
  auto q_slot = [](int) { return 0; };
  auto do_slot = [](int) { return 1; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
      mbar_init(bar_vec_full(i), 1);
      mbar_init(bar_vec_empty(i), 256);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_read, 256);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_ready, 256);
    mbar_init(bar_k_tmem, 256);
    mbar_init(bar_o_final, 1);
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

  if (warp == kWProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_do);
      mbar_arrive_expect_tx(bar_kv_full, 2 * kWTile);
      for (int bx = 0; bx < kWD / 64; ++bx) {
        tma_load_3d(s_k + bx * kBoxBytes, &map_k, bar_kv_full, bx * 64, jt * kBN, bhkv);
        tma_load_3d(s_v + bx * kBoxBytes, &map_v, bar_kv_full, bx * 64, jt * kBN, bhkv);
      }
      int uses[2] = {0, 0};
      auto load = [&](const CUtensorMap* m, int slot, int row0, int bh) -> bool {
        // slot 0 takes Q/dO only once every row of K is in TMEM
        if (slot == 0 && uses[0] == 0 && !mbar_wait(bar_k_tmem, 0, abort_flag, deadline)) return false;
        if (!mbar_wait(bar_empty(slot), (uses[slot] & 1) ^ 1, abort_flag, deadline)) return false;
        ++uses[slot];
        mbar_arrive_expect_tx(bar_full(slot), kWTile);
        for (int bx = 0; bx < kWD / 64; ++bx)
          tma_load_3d(s_slot(slot) + bx * kBoxBytes, m, bar_full(slot), bx * 64, row0, bh);
        return true;
      };
      for (int t = 0; t < nsteps; ++t) {
        const int bh = step_head(t), row0 = step_tile(t) * kBM;
        if (!load(&map_do, do_slot(t), row0, bh)) break;
        if (!load(&map_q, q_slot(t), row0, bh)) break;
        const int vb = t & 1;
        if (!mbar_wait(bar_vec_empty(vb), ((t >> 1) & 1) ^ 1, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_vec_full(vb), 2 * kBM * 4);
        const size_t voff = static_cast<size_t>(bh) * p.NQP + row0;
        bulk_load(s_vec(vb), p.ws_lse2 + voff, kBM * 4, bar_vec_full(vb));
        bulk_load(s_vec(vb) + kBM * 4, p.ws_d + voff, kBM * 4, bar_vec_full(vb));
      }
    }
    __syncwarp();
  } else if (warp == kWIss) {
    // ------------------------------------------------------------ MMA issuer
    // dP^T_0; per step t: [dP^T_t read] S^T_t into the same columns, [dS^T_t
    // written] dK_t (Q_t's slot free after), [dO_{t+1}] dP^T_{t+1} (dO_t's slot
    // was free once dP^T_t completed).
    if (lane == 0) {
      int fulls[2] = {0, 0};
      auto wait_full = [&](int slot) -> bool {
        return mbar_wait(bar_full(slot), (fulls[slot]++) & 1, abort_flag, deadline);
      };
      bool ok = !p.test_stall || mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      ok = ok && (nsteps == 0 || (mbar_wait(bar_kv_full, 0, abort_flag, deadline) &&
                                  mbar_wait(bar_k_tmem, 0, abort_flag, deadline)));
      const uint32_t id_s = make_idesc(1, 128, 128, 0, 0);     // S^T, dP^T: K-major operands
      const uint32_t id_k = make_idesc(1, 128, kWD, 0, 1);     // dK: A = dS^T K-major, B = Q MN-major
      auto scores = [&](int t) {     // S^T_t = K Q_t^T, A = K from TMEM
        const uint64_t qd = smem_desc_sw128(s_slot(q_slot(t)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ts(tbase + C::kColSP, tbase + C::kColK + kk * 8, desc_add(qd, off), id_s, kk > 0);
        }
        mma_commit(bar_s_full);
      };
      auto dp = [&](int t) {         // dP^T_t = V dO_t^T
        const uint64_t vd = smem_desc_sw128(s_v, 16, 1024), dod = smem_desc_sw128(s_slot(do_slot(t)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColSP, desc_add(vd, off), desc_add(dod, off), id_s, kk > 0);
        }
        mma_commit(bar_dp_full);
        mma_commit(bar_empty(do_slot(t)));
      };
      auto dk = [&](int t) {         // dK += dS^T Q_t over the step's 128 queries
        const uint64_t dsd = smem_desc_sw128(s_ds, 16, 1024);
        const uint64_t qmn = smem_desc_sw128(s_slot(q_slot(t)), kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + kWColAcc, desc_add(dsd, off), desc_add(qmn, kk * 16 * 128), id_k, t > 0 || kk > 0);
        }
        mma_commit(bar_empty(q_slot(t)));
      };
      if (ok && nsteps > 0) {
        ok = wait_full(do_slot(0));
        if (ok) {
          tc_fence_after();
          dp(0);
        }
      }
      for (int t = 0; t < nsteps && ok; ++t) {
        if (!(ok = mbar_wait(bar_s_read, t & 1, abort_flag, deadline))) break;   // every warp read dP^T_t
        if (!(ok = wait_full(q_slot(t)))) break;
        tc_fence_after();
        scores(t);
        // the single dS^T buffer: dS^T_t is written after S^T_t completes, so
        // after dK_{t-1} (issued before S^T_t) has read dS^T_{t-1}
        if (!(ok = mbar_wait(bar_ready, t & 1, abort_flag, deadline))) break;
        tc_fence_after();
        dk(t);
        if (t + 1 < nsteps) {
          // the score columns: every warp read S^T_t before its dS^T_t
          if (!(ok = wait_full(do_slot(t + 1)))) break;
          tc_fence_after();
          dp(t + 1);
        }
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ one thread per key row and column half
    const int quarter = warp & 3, g = warp >> 2;   // g: queries [64g, 64g + 64) of each step
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int key = jt * kBN + r;
    const bool key_pad = key >= p.Nk;
    const float sl2 = p.scale_log2;
    const uint32_t t_sp = tbase + lane_off + C::kColSP;
    bool ok = true;
    if (nsteps > 0) {
      // this key row of K into TMEM as the A operand of S^T (128 columns of
      // bf16 pairs, the tile's 16-byte units in order; this warp's two boxes);
      // slot 0 is then free
      ok = mbar_wait(bar_kv_full, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
#pragma unroll
        for (int bx = 2 * g; bx < 2 * g + 2; ++bx) {
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4 * u]), "=r"(w[4 * u + 1]), "=r"(w[4 * u + 2]), "=r"(w[4 * u + 3])
                         : "r"(swz128(s_k + bx * kBoxBytes, r, u)));
          tmem_st_32x32b_x32(tbase + lane_off + C::kColK + 32u * bx, w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_k_tmem);
      }
    }
    for (int t = 0; t < nsteps && ok; ++t) {
      const int vb = t & 1;
      ok = mbar_wait(bar_dp_full, t & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float dpv[64];
      tmem_ld64(t_sp + 64u * g, dpv);
      // dP^T_t is in registers: its columns may take S^T_t
      tc_fence_before();
      mbar_arrive(bar_s_read);
      ok = mbar_wait(bar_s_full, t & 1, abort_flag, deadline) &&
           mbar_wait(bar_vec_full(vb), (t >> 1) & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* vec = reinterpret_cast<const float*>(gbase + (s_vec(vb) - base)) + 64 * g;
      {
        // P^T[key, q] = 2^(S^T s log2e - LSE_q log2e); causal: q + (Nk - N) >= key;
        // dS^T = P^T (dP^T - D), formed in dpv in place, 32 columns of S^T at a time
        const int lim = key - p.causal_off - step_tile(t) * kBM - 64 * g;   // first visible column of the half
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t sr[32];
          tmem_ld_32x32b_x32(t_sp + 64 * g + 32 * h, sr);
          tmem_wait_ld();
          reg_fence_x32(sr);
#pragma unroll
          for (int c = 32 * h; c < 32 * h + 32; ++c) {
            const float e = ex2_approx(fmaf(__uint_as_float(sr[c & 31]), sl2, -vec[c]));
            const float pr = (key_pad || (p.causal && c < lim)) ? 0.f : e;
            dpv[c] = pr * (dpv[c] - vec[kBM + c]);
          }
        }
        // dS^T row r, queries [64 g, 64 g + 64): box g
        store_row64(s_ds + g * kBoxBytes, r, dpv);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_ready);
      mbar_arrive(bar_vec_empty(vb));
    }
    // ---------------------------------------------------------- epilogue
    if (ok) {
      ok = mbar_wait(bar_o_final, 0, abort_flag, deadline);
      if (nsteps == 0) ok = ok && mbar_wait(bar_kv_full, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    // staging: the V tile, idle once every MMA has completed
    const uint32_t stg = s_v;
    if (ok) {
      tc_fence_after();
      if (nsteps > 0) {
        stage_acc_row(tbase + lane_off + kWColAcc, stg, r, p.scale, g);
      } else {
#pragma unroll
        for (int bx = 2 * g; bx < 2 * g + 2; ++bx)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" :: "r"(swz128(stg + bx * kBoxBytes, r, u)), "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (!*abort_flag && warp == 0 && lane == 0 && jt < nkt) {
      for (int bx = 0; bx < kWD / 64; ++bx) tma_store_3d(&map_dk, stg + bx * kBoxBytes, bx * 64, jt * kBN, bhkv);
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

// ------------------------------------------------------------------ dV per key tile, 128-query steps
// Shared memory: K (one [128, 256] bf16 tile) | a ring of four 32 KB slots |
// LSE x3 | barriers. Every Q and dO tile travels through the ring as two
// pieces of 128 columns (two 64-column boxes each), in the order the products
// read them: Q_0, Q_1, then per step t dO_t and Q_{t+2}. A tile's two pieces
// always take slots 0-1 or 2-3, so one N = 256 product group can read dO_t
// across both. A slot goes back to the producer when the products that read
// its piece complete, so loads run up to four pieces (one step) ahead of the
// tensor core.
// TMEM: dV accumulator | S^T buffer 0 | S^T buffer 1 (128 columns each).
// Products: S^T_0 and S^T_1, then per step t [P^T_t written] dV_t (N = 256
// over both dO pieces) and S^T_{t+2} into the buffer dV_t has
// just read, so the warps form P^T_{t+1} while the tensor core runs dV_t and
// S^T_{t+2}. With 128 queries per step S^T = K Q^T is an N = 128 product (an
// N = 64 product takes about as long).
struct WideDvCfg {
  static constexpr int kOffK = 0;
  static constexpr int kSlots = 4;
  static constexpr int kSlotBytes = 2 * kBoxBytes;     // [128, 128] bf16: half of a Q or dO tile
  static constexpr int kOffRing = kWTile;
  static constexpr int kNVec = 3;                      // LSE buffers: step t in buffer t % 3
  static constexpr int kVecBytes = 512;                // LSE log2(e) of 128 queries
  static constexpr int kOffVec = kOffRing + kSlots * kSlotBytes;
  static constexpr int kOffBar = kOffVec + kNVec * kVecBytes;
  static constexpr int kLayout = kOffBar + 256;
  static constexpr int kSmemAlloc = kLayout + 1024;
  static constexpr uint32_t kColS = 256;               // buffers at 256 and 384
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(kWThreads, 1)
wide_dv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_do, const __grid_constant__ CUtensorMap map_dv,
               const BwdParams p) {
  using C = WideDvCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  if ((base - raw) + C::kLayout > static_cast<uint32_t>(C::kSmemAlloc)) {
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  const uint32_t s_k = base + C::kOffK;
  auto s_slot = [&](int i) { return base + C::kOffRing + i * C::kSlotBytes; };
  auto s_vec = [&](int i) { return base + C::kOffVec + i * C::kVecBytes; };
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_k_full = bars;
  auto bar_full = [&](int i) { return bars + 8u + 8u * i; };           // ring slot i landed
  auto bar_empty = [&](int i) { return bars + 48u + 8u * i; };         // ring slot i read
  auto bar_vec_full = [&](int i) { return bars + 88u + 8u * i; };
  auto bar_vec_empty = [&](int i) { return bars + 112u + 8u * i; };
  auto bar_s_full = [&](int i) { return bars + 136u + 8u * i; };
  auto bar_ready = [&](int i) { return bars + 152u + 8u * i; };      // P^T written over S^T
  const uint32_t bar_o_final = bars + 168, bar_stall = bars + 176;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 184);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 188);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (key tile, batch * kv head), KV heads in groups of
  // p.head_group, small key tiles first (the most query tiles when causal)
  const int nkt = p.NKP / kBN;
  const int grp = blockIdx.x / (nkt * p.head_group);
  const int gsize = min(p.head_group, p.BHkv - grp * p.head_group);
  const int local = blockIdx.x - grp * p.head_group * nkt;
  const int jt = local / gsize;
  const int bhkv = grp * p.head_group + local % gsize;
  const int b = bhkv / p.Hkv, hk = bhkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int nq = p.NQP / kBM;
  // first query tile that sees key tile jt (bottom-right causal)
  const int first_row = jt * kBN - p.causal_off;
  const int it0 = p.causal ? (first_row <= 0 ? 0 : min(nq, first_row / kBM)) : 0;
  const int per_head = nq - it0;
  const int nsteps = G * per_head;
  auto step_head = [&](int t) { return b * p.Hq + hk * G + t / per_head; };
  auto step_tile = [&](int t) { return it0 + t % per_head; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_k_full, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int i = 0; i < C::kNVec; ++i) {
      mbar_init(bar_vec_full(i), 1);
      mbar_init(bar_vec_empty(i), 256);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_ready(i), 256);
    }
    mbar_init(bar_o_final, 1);
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

  if (warp == kWProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_do);
      mbar_arrive_expect_tx(bar_k_full, kWTile);
      for (int bx = 0; bx < kWD / 64; ++bx)
        tma_load_3d(s_k + bx * kBoxBytes, &map_k, bar_k_full, bx * 64, jt * kBN, bhkv);
      int k = 0;                                       // ring pieces issued
      // columns [128 half, 128 half + 128) of rows [row0, row0 + 128) of head bh
      auto piece = [&](const CUtensorMap* m, int row0, int bh, int half) -> bool {
        const int slot = k % C::kSlots, use = k / C::kSlots;
        ++k;
        if (!mbar_wait(bar_empty(slot), (use & 1) ^ 1, abort_flag, deadline)) return false;
        mbar_arrive_expect_tx(bar_full(slot), C::kSlotBytes);
        for (int bx = 0; bx < 2; ++bx)
          tma_load_3d(s_slot(slot) + bx * kBoxBytes, m, bar_full(slot), (2 * half + bx) * 64, row0, bh);
        return true;
      };
      auto load_q = [&](int t) -> bool {              // Q_t and the LSE of step t
        const int bh = step_head(t), it = step_tile(t), vb = t % C::kNVec;
        if (!mbar_wait(bar_vec_empty(vb), ((t / C::kNVec) & 1) ^ 1, abort_flag, deadline)) return false;
        mbar_arrive_expect_tx(bar_vec_full(vb), C::kVecBytes);
        bulk_load(s_vec(vb), p.ws_lse2 + static_cast<size_t>(bh) * p.NQP + static_cast<size_t>(it) * kBM, C::kVecBytes,
                  bar_vec_full(vb));
        return piece(&map_q, it * kBM, bh, 0) && piece(&map_q, it * kBM, bh, 1);
      };
      bool ok = (nsteps < 1 || load_q(0)) && (nsteps < 2 || load_q(1));
      for (int t = 0; t < nsteps && ok; ++t) {
        const int bh = step_head(t), row0 = step_tile(t) * kBM;
        ok = piece(&map_do, row0, bh, 0) && piece(&map_do, row0, bh, 1);
        if (ok && t + 2 < nsteps) ok = load_q(t + 2);
      }
    }
    __syncwarp();
  } else if (warp == kWIss) {
    // ------------------------------------------------------------ MMA issuer
    // S^T_0, S^T_1; per step t: [P^T_t written] dV_t, then S^T_{t+2} into the
    // buffer dV_t has read. Each piece is taken from the ring in the order the
    // producer loads it and handed back by a commit after its products.
    if (lane == 0) {
      bool ok = !p.test_stall || mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      ok = ok && (nsteps == 0 || mbar_wait(bar_k_full, 0, abort_flag, deadline));
      const uint32_t id_s = make_idesc(1, 128, 128, 0, 0);     // S^T: K and Q both K-major
      const uint32_t id_v = make_idesc(1, 128, kWD, 0, 1);     // dV: A = P^T from TMEM, B = dO MN-major
      const uint64_t kd = smem_desc_sw128(s_k, 16, 1024);
      const uint64_t ring_k = smem_desc_sw128(s_slot(0), 16, 1024);           // K-major view of slot 0
      const uint64_t ring_mn = smem_desc_sw128(s_slot(0), kBoxBytes, 1024);   // MN-major view of slot 0
      int k = 0;                                       // ring pieces taken
      auto take = [&](int& slot) -> bool {
        slot = k % C::kSlots;
        const int use = k / C::kSlots;
        ++k;
        if (!mbar_wait(bar_full(slot), use & 1, abort_flag, deadline)) return false;
        tc_fence_after();
        return true;
      };
      auto scores = [&](int t) -> bool {              // S^T_t = K Q_t^T, the two halves of d in turn
        const uint32_t d = tbase + C::kColS + 128u * (t & 1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          int slot;
          if (!take(slot)) return false;
          const uint64_t qd = desc_add(ring_k, static_cast<uint32_t>(slot * C::kSlotBytes));
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {
            const int kk = 8 * h + k8;
            const uint32_t off_k = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
            const uint32_t off_q = (k8 * 32 / 128) * kBoxBytes + (k8 * 32) % 128;
            mma_bf16_ss(d, desc_add(kd, off_k), desc_add(qd, off_q), id_s, kk > 0);
          }
          mma_commit(bar_empty(slot));
        }
        mma_commit(bar_s_full(t & 1));
        return true;
      };
      auto dv = [&](int t) -> bool {                  // dV += P^T dO_t (K = 128 queries), d in two halves
        const uint32_t a = tbase + C::kColS + 128u * (t & 1);
        int s0, s1;                                    // adjacent slots: pieces come in pairs from an even slot
        if (!take(s0) || !take(s1)) return false;
        const uint64_t dod = desc_add(ring_mn, static_cast<uint32_t>(s0 * C::kSlotBytes));
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          mma_bf16_ts(tbase + kWColAcc, a + 64 * (kk >> 2) + (kk & 3) * 8, desc_add(dod, kk * 16 * 128), id_v,
                      t > 0 || kk > 0);
        mma_commit(bar_empty(s0));
        mma_commit(bar_empty(s1));
        return true;
      };
      ok = ok && (nsteps < 1 || scores(0)) && (nsteps < 2 || scores(1));
      for (int t = 0; t < nsteps && ok; ++t) {
        if (!(ok = mbar_wait(bar_ready(t & 1), (t >> 1) & 1, abort_flag, deadline))) break;
        tc_fence_after();
        ok = dv(t);
        // S^T_{t+2} goes into the buffer whose P^T_t dV_t (issued before) reads
        if (ok && t + 2 < nsteps) ok = scores(t + 2);
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ one thread per key row and column half
    const int quarter = warp & 3, g = warp >> 2;   // g: queries [64g, 64g + 64) of each step
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int key = jt * kBN + r;
    const bool key_pad = key >= p.Nk;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < nsteps && ok; ++t) {
      const int sb = t & 1, vb = t % C::kNVec;
      ok = mbar_wait(bar_s_full(sb), (t >> 1) & 1, abort_flag, deadline) &&
           mbar_wait(bar_vec_full(vb), (t / C::kNVec) & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(gbase + (s_vec(vb) - base)) + 64 * g;
      const uint32_t ts = tbase + lane_off + C::kColS + 128u * sb + 64u * g;
      uint32_t sr[2][32];
      tmem_ld_32x32b_x32(ts, sr[0]);
      tmem_ld_32x32b_x32(ts + 32, sr[1]);
      tmem_wait_ld();
      reg_fence_x32(sr[0]);
      reg_fence_x32(sr[1]);
      // P^T[key, q] = 2^(S^T s log2e - LSE_q log2e); causal: q + (Nk - N) >= key;
      // query rows past N have LSE = +inf, so P = 0
      const int lim = key - p.causal_off - step_tile(t) * kBM - 64 * g;   // first visible column of the half
      uint32_t pp[32];
#pragma unroll
      for (int c2 = 0; c2 < 32; ++c2) {
        float e[2];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int c = 2 * c2 + e2;
          const float pe = ex2_approx(fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, -lse2[c]));
          e[e2] = (key_pad || (p.causal && c < lim)) ? 0.f : pe;
        }
        pp[c2] = pack_bf16x2(e[0], e[1]);
      }
      // P^T over the first 32 of the S^T columns this thread has read: queries
      // 64g + 2c2, +1 in column 64g + c2
      tmem_st_32x32b_x32(ts, pp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ready(sb));
      mbar_arrive(bar_vec_empty(vb));
    }
    // ---------------------------------------------------------- epilogue
    if (ok) {
      ok = mbar_wait(bar_o_final, 0, abort_flag, deadline);
      if (nsteps == 0) ok = ok && mbar_wait(bar_k_full, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    // staging: the K tile, idle once every MMA has completed
    if (ok) {
      tc_fence_after();
      if (nsteps > 0) {
        stage_acc_row(tbase + lane_off + kWColAcc, s_k, r, 1.0f, g);
      } else {
#pragma unroll
        for (int bx = 2 * g; bx < 2 * g + 2; ++bx)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" :: "r"(swz128(s_k + bx * kBoxBytes, r, u)), "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (!*abort_flag && warp == 0 && lane == 0) {
      for (int bx = 0; bx < kWD / 64; ++bx) tma_store_3d(&map_dv, s_k + bx * kBoxBytes, bx * 64, jt * kBN, bhkv);
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

// ------------------------------------------------------------------ dQ per query tile, 128-key steps
// Shared memory: dO | two 64 KB slots | dS | barriers. Q lands in slot 0 and
// the warps copy it into TMEM as the A operand of S; K_j then always goes to
// slot 0 and V_j to slot 1, so V_{j+1} loads as soon as dP_j has read V_j,
// early in step j, and K_{j+1} once dQ_j has read K_j.
// TMEM: dQ accumulator | dP, then S, of the step (128 columns) | Q.
// Per step dP_j (N = 128 keys) goes into the score columns; once every warp
// has read it into registers, S_j goes into the same columns; once every
// warp has written dS_j, dQ_j += dS_j K_j, and dP_{j+1} follows. With 128
// keys per step every score product is N = 128 (an N = 64 product takes
// about as long).
struct WideDqCfg {
  static constexpr int kOffDo = 0;
  static constexpr int kOffSlot = kWTile;              // two 64 KB slots; slot 0 first holds Q
  static constexpr int kOffDs = kOffSlot + 2 * kWTile;  // dS [128 queries, 128 keys] bf16: two boxes
  static constexpr int kOffBar = kOffDs + 2 * kBoxBytes;
  static constexpr uint32_t kColSP = 256, kColQ = 384;
  static constexpr int kLayout = kOffBar + 256;
  static constexpr int kSmemAlloc = kLayout + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(kWThreads, 1)
wide_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
               const __grid_constant__ CUtensorMap map_dq, const BwdParams p) {
  using C = WideDqCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  if ((base - raw) + C::kLayout > static_cast<uint32_t>(C::kSmemAlloc)) {
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  const uint32_t s_do = base + C::kOffDo;
  auto s_slot = [&](int i) { return base + C::kOffSlot + i * kWTile; };
  const uint32_t s_q = s_slot(0);                      // the Q tile, then the dQ staging
  const uint32_t s_ds = base + C::kOffDs;
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_q_full = bars;                    // Q and dO landed
  auto bar_full = [&](int i) { return bars + 8u + 8u * i; };
  auto bar_empty = [&](int i) { return bars + 24u + 8u * i; };
  const uint32_t bar_s_full = bars + 40, bar_s_read = bars + 48, bar_dp_full = bars + 56;
  const uint32_t bar_ready = bars + 64, bar_o_final = bars + 72, bar_stall = bars + 80;
  const uint32_t bar_q_tmem = bars + 88;               // every row of Q copied into TMEM
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 96);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 100);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (query tile, batch * head); causal: the longest rows first.
  // Query heads go in groups of p.head_group whose K and V fit in part of L2.
  const int nq = p.NQP / kBM;
  const int grp = blockIdx.x / (nq * p.head_group);
  const int gsize = min(p.head_group, p.BH - grp * p.head_group);
  const int local = blockIdx.x - grp * p.head_group * nq;
  const int qt = nq - 1 - local / gsize;
  const int bh = grp * p.head_group + local % gsize;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bh_kv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int nkt = p.NKP / kBN;
  int nsteps = nkt;
  if (p.causal) {
    const int last = qt * kBM + kBM - 1 + p.causal_off;   // the tile's last row sees keys up to here
    nsteps = last < 0 ? 0 : min(nkt, last / kBN + 1);
  }
  // K_j always in slot 0 (after Q has gone from it into TMEM), V_j in slot 1:
  // V_{j+1} loads as soon as dP_j has read V_j, early in step j
  auto k_slot = [](int) { return 0; };
  auto v_slot = [](int) { return 1; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_read, 256);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_ready, 256);
    mbar_init(bar_q_tmem, 256);
    mbar_init(bar_o_final, 1);
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

  if (warp == kWProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nsteps > 0) {
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      mbar_arrive_expect_tx(bar_q_full, 2 * kWTile);
      for (int bx = 0; bx < kWD / 64; ++bx) {
        tma_load_3d(s_q + bx * kBoxBytes, &map_q, bar_q_full, bx * 64, qt * kBM, bh);
        tma_load_3d(s_do + bx * kBoxBytes, &map_do, bar_q_full, bx * 64, qt * kBM, bh);
      }
      int uses[2] = {0, 0};
      auto load = [&](const CUtensorMap* m, int slot, int row0) -> bool {
        // slot 0 takes K/V only once every row of Q is in TMEM
        if (slot == 0 && uses[0] == 0 && !mbar_wait(bar_q_tmem, 0, abort_flag, deadline)) return false;
        if (!mbar_wait(bar_empty(slot), (uses[slot] & 1) ^ 1, abort_flag, deadline)) return false;
        ++uses[slot];
        mbar_arrive_expect_tx(bar_full(slot), kWTile);
        for (int bx = 0; bx < kWD / 64; ++bx)
          tma_load_3d(s_slot(slot) + bx * kBoxBytes, m, bar_full(slot), bx * 64, row0, bh_kv);
        return true;
      };
      for (int j = 0; j < nsteps; ++j) {
        if (!load(&map_v, v_slot(j), j * kBN)) break;
        if (!load(&map_k, k_slot(j), j * kBN)) break;
      }
    }
    __syncwarp();
  } else if (warp == kWIss) {
    // ------------------------------------------------------------ MMA issuer
    // dP_0; per step j: [dP_j read] S_j into the same columns, [dS_j written]
    // dQ_j (K_j's slot free after), [V_{j+1}] dP_{j+1} (V_j's slot was free
    // once dP_j completed).
    if (lane == 0) {
      int fulls[2] = {0, 0};
      auto wait_full = [&](int slot) -> bool {
        return mbar_wait(bar_full(slot), (fulls[slot]++) & 1, abort_flag, deadline);
      };
      bool ok = !p.test_stall || mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      ok = ok && (nsteps == 0 || (mbar_wait(bar_q_full, 0, abort_flag, deadline) &&
                                  mbar_wait(bar_q_tmem, 0, abort_flag, deadline)));
      const uint32_t id_s = make_idesc(1, 128, 128, 0, 0);     // S, dP: K-major operands
      const uint32_t id_q = make_idesc(1, 128, kWD, 0, 1);     // dQ: A = dS K-major, B = K MN-major
      auto scores = [&](int j) {     // S_j = Q K_j^T, A = Q from TMEM
        const uint64_t kd = smem_desc_sw128(s_slot(k_slot(j)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ts(tbase + C::kColSP, tbase + C::kColQ + kk * 8, desc_add(kd, off), id_s, kk > 0);
        }
        mma_commit(bar_s_full);
      };
      auto dp = [&](int j) {         // dP_j = dO V_j^T
        const uint64_t dod = smem_desc_sw128(s_do, 16, 1024), vd = smem_desc_sw128(s_slot(v_slot(j)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColSP, desc_add(dod, off), desc_add(vd, off), id_s, kk > 0);
        }
        mma_commit(bar_dp_full);
        mma_commit(bar_empty(v_slot(j)));
      };
      auto dq = [&](int j) {         // dQ += dS K_j over the step's 128 keys
        const uint64_t dsd = smem_desc_sw128(s_ds, 16, 1024);
        const uint64_t kmn = smem_desc_sw128(s_slot(k_slot(j)), kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + kWColAcc, desc_add(dsd, off), desc_add(kmn, kk * 16 * 128), id_q, j > 0 || kk > 0);
        }
        mma_commit(bar_empty(k_slot(j)));
      };
      if (ok && nsteps > 0) {
        ok = wait_full(v_slot(0));
        if (ok) {
          tc_fence_after();
          dp(0);
        }
      }
      for (int j = 0; j < nsteps && ok; ++j) {
        if (!(ok = mbar_wait(bar_s_read, j & 1, abort_flag, deadline))) break;   // every warp read dP_j
        if (!(ok = wait_full(k_slot(j)))) break;
        tc_fence_after();
        scores(j);
        // the single dS buffer: dS_j is written after S_j completes, so after
        // dQ_{j-1} (issued before S_j) has read dS_{j-1}
        if (!(ok = mbar_wait(bar_ready, j & 1, abort_flag, deadline))) break;
        tc_fence_after();
        dq(j);
        if (j + 1 < nsteps) {
          // the score columns: every warp read S_j before its dS_j
          if (!(ok = wait_full(v_slot(j + 1)))) break;
          tc_fence_after();
          dp(j + 1);
        }
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ one thread per query row and column half
    const int quarter = warp & 3, g = warp >> 2;   // g: keys [64g, 64g + 64) of each step
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int q = qt * kBM + r;
    const float sl2 = p.scale_log2;
    // this row's LSE log2(e) (+inf past N: P = 0) and D
    const float lse2 = p.ws_lse2[static_cast<size_t>(bh) * p.NQP + qt * kBM + r];
    const float dsub = p.ws_d[static_cast<size_t>(bh) * p.NQP + qt * kBM + r];
    const int key_lim = p.causal ? min(p.Nk, q + p.causal_off + 1) : p.Nk;   // keys < key_lim are visible
    const uint32_t t_sp = tbase + lane_off + C::kColSP;
    bool ok = true;
    if (nsteps > 0) {
      // this row of Q into TMEM as the A operand of S: 128 columns of bf16
      // pairs, the lower dimension in the low half (the tile's 16-byte units
      // in order; this warp's two boxes); slot 0 is then free for K and V
      ok = mbar_wait(bar_q_full, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
#pragma unroll
        for (int bx = 2 * g; bx < 2 * g + 2; ++bx) {
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4 * u]), "=r"(w[4 * u + 1]), "=r"(w[4 * u + 2]), "=r"(w[4 * u + 3])
                         : "r"(swz128(s_q + bx * kBoxBytes, r, u)));
          tmem_st_32x32b_x32(tbase + lane_off + C::kColQ + 32u * bx, w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_q_tmem);
      }
    }
    for (int j = 0; j < nsteps && ok; ++j) {
      ok = mbar_wait(bar_dp_full, j & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float dpv[64];
      tmem_ld64(t_sp + 64u * g, dpv);
      // dP_j is in registers: its columns may take S_j
      tc_fence_before();
      mbar_arrive(bar_s_read);
      ok = mbar_wait(bar_s_full, j & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t sr[2][32];
        tmem_ld_32x32b_x32(t_sp + 64 * g, sr[0]);
        tmem_ld_32x32b_x32(t_sp + 64 * g + 32, sr[1]);
        tmem_wait_ld();
        reg_fence_x32(sr[0]);
        reg_fence_x32(sr[1]);
        // P = 2^(S s log2e - LSE log2e), dS = P (dP - D)
        const int lim = key_lim - j * kBN - 64 * g;
#pragma unroll
        for (int c = 0; c < 64; ++c) {                  // dpv becomes dS in place
          const float pe = ex2_approx(fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, -lse2));
          const float pr = (c < lim) ? pe : 0.f;
          dpv[c] = pr * (dpv[c] - dsub);
        }
        // dS row r, keys [64 g, 64 g + 64): box g
        store_row64(s_ds + g * kBoxBytes, r, dpv);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_ready);
    }
    // ---------------------------------------------------------- epilogue
    if (ok) {
      ok = mbar_wait(bar_o_final, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      // staging: the Q tile, idle once every MMA has completed
      if (nsteps > 0) {
        stage_acc_row(tbase + lane_off + kWColAcc, s_q, r, p.scale, g);
      } else {
#pragma unroll
        for (int bx = 2 * g; bx < 2 * g + 2; ++bx)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" :: "r"(swz128(s_q + bx * kBoxBytes, r, u)), "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (!*abort_flag && warp == 0 && lane == 0) {
      for (int bx = 0; bx < kWD / 64; ++bx) tma_store_3d(&map_dq, s_q + bx * kBoxBytes, bx * 64, qt * kBM, bh);
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

// ------------------------------------------------------------------ launch
cudaError_t launch_bwd_wide(const BwdMaps& m, const BwdMaps& m64, const BwdParams& p, cudaStream_t stream) {
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    cudaError_t r = cudaFuncSetAttribute(wide_dv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         WideDvCfg::kSmemAlloc);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(wide_dk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WideDkCfg::kSmemAlloc);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(wide_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WideDqCfg::kSmemAlloc);
    return r;
  });
  if (e != cudaSuccess) return e;
  const int kv_grid = (p.NKP / kBN) * p.BHkv;
  const int q_grid = (p.NQP / kBM) * p.BH;
  // head groups whose streamed operands (bf16) fit in 64 MB, half of L2: the kv
  // passes stream the Q and dO of a KV head's G query heads, the dQ pass the K
  // and V of a query head's KV head (shared by its G siblings, kept adjacent)
  const long long G = p.Hq / p.Hkv;
  const long long budget = 64LL << 20;
  BwdParams pk = p, pq = p;
  pk.head_group = static_cast<int>(std::max(1LL, std::min<long long>(p.BHkv, budget / (4LL * G * p.N * kWD))));
  pq.head_group = static_cast<int>(std::max(1LL, std::min<long long>(p.BH, budget * G / (4LL * p.Nk * kWD))));
  wide_dv_kernel<<<kv_grid, kWThreads, WideDvCfg::kSmemAlloc, stream>>>(m.q, m.k, m.dO, m.dv, pk);
  cudaError_t r = cudaGetLastError();
  if (r != cudaSuccess) return r;
  wide_dk_kernel<<<kv_grid, kWThreads, WideDkCfg::kSmemAlloc, stream>>>(m.q, m.k, m.v, m.dO, m.dk, pk);
  r = cudaGetLastError();
  if (r != cudaSuccess) return r;
  wide_dq_kernel<<<q_grid, kWThreads, WideDqCfg::kSmemAlloc, stream>>>(m.q, m.k, m.v, m.dO, m.dq, pq);
  return cudaGetLastError();
}

}  // namespace fa
