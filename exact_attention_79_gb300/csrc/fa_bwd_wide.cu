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
// memory. The gradients are therefore formed in three passes, each with a
// fixed order of additions (no atomics: every output is bit reproducible):
//   wide_dv_kernel  per 128-key tile: S^T = K Q_t^T (N = 128 queries),
//                   P^T -> TMEM (bf16), dV += P^T dO_t          over 128-query steps t
//   wide_dk_kernel  per 128-key tile: S^T, dP^T = V dO_s^T over 64-query
//                   sub-tiles, dS^T = P^T (dP^T - D) -> shared memory, dK += dS^T Q_s
//   wide_dq_kernel  per 128-row query tile: S = Q K_j^T, dP = dO V_j^T over
//                   64-key sub-tiles, dS -> shared memory, dQ += dS K_j
// S (or S^T) and dP are formed twice or three times: 8 GEMMs of the 5 the
// method needs. bwd_pre_kernel (fa_bwd.cu) writes D and the base-2 LSE first.
// The dK and dQ passes keep K or Q in TMEM as the A operand of the scores and
// stream the other operands through a ring of four 32 KB slots.
//
// Roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA issuer
// (one thread), warps 2-5 one thread per TMEM lane (key row in the dV and dK
// passes, query row in the dQ pass).
#include <algorithm>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kWD = 256;                          // head-dimension build
constexpr int kWSub = 64;                         // rows of a sub-tile step
constexpr int kWTile = kWD / 64 * kBoxBytes;      // [128, 256] bf16: 64 KB
constexpr int kWSubTile = kWTile / 2;             // [64, 256] bf16: 32 KB
constexpr int kWSubBox = kBoxBytes / 2;           // one 64-row box: 8 KB
constexpr int kWDs = kBoxBytes;                   // [128, 64] bf16 (dS or dS^T): 16 KB
constexpr int kWThreads = 192;
constexpr uint32_t kWColAcc = 0, kWColS = 256;   // TMEM: accumulator (256 columns) | scores

// S (M = 128 rows of `a`, N = 64 rows of `b`, K = 256): both K-major, `a` in
// boxes of 128 rows (16 KB), `b` in boxes of 64 rows (8 KB)
__device__ __forceinline__ void issue_scores(uint32_t d_tmem, uint32_t a, uint32_t b) {
  const uint32_t id = make_idesc(1, 128, kWSub, 0, 0);
  const uint64_t ad = smem_desc_sw128(a, 16, 1024), bd = smem_desc_sw128(b, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < kWD / 16; ++kk) {
    const uint32_t kb = kk * 32;
    mma_bf16_ss(d_tmem, desc_add(ad, (kb / 128) * kBoxBytes + kb % 128),
                desc_add(bd, (kb / 128) * kWSubBox + kb % 128), id, kk > 0);
  }
}

// D[128, 256] += A[128, 64] B[64, 256]: B MN-major in boxes of 64 rows (one box
// per 64 columns); A K-major in shared memory (one 16 KB box) or in TMEM
__device__ __forceinline__ void issue_acc_ss(uint32_t d_tmem, uint32_t a, uint32_t b, bool acc) {
  const uint32_t id = make_idesc(1, 128, kWD, 0, 1);
  const uint64_t ad = smem_desc_sw128(a, 16, 1024), bd = smem_desc_sw128(b, kWSubBox, 1024);
#pragma unroll
  for (int kk = 0; kk < kWSub / 16; ++kk)
    mma_bf16_ss(d_tmem, desc_add(ad, kk * 32), desc_add(bd, kk * 16 * 128), id, acc || kk > 0);
}
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

// The 256 fp32 accumulator columns of this thread's lane, times `mul`, as
// row `row` of a [128, 256] bf16 tile (four 128-row boxes) at `stg`
__device__ __forceinline__ void stage_acc_row(uint32_t taddr, uint32_t stg, int row, float mul) {
#pragma unroll
  for (int c0 = 0; c0 < kWD; c0 += 32) {
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

// ------------------------------------------------------------------ dK per key tile
// Shared memory: V | four 32 KB slots | dS^T x2 | LSE, D x2 | barriers. K
// lands in slots 0 and 1, the warps copy it into TMEM as the A operand of
// S^T, and the slots then join a ring in which Q_s and dO_s are items 2s and
// 2s+1 in slot (item + 2) % 4.
struct WideDkCfg {
  static constexpr int kSlots = 4;
  static constexpr int kOffV = 0;
  static constexpr int kOffSlot = kWTile;
  static constexpr int kOffK = kOffSlot;                                // slots 0-1, then TMEM
  static constexpr int kOffDs = kOffSlot + kSlots * kWSubTile;
  static constexpr int kOffVec = kOffDs + 2 * kWDs;
  static constexpr int kVecBytes = 512;                                 // LSE[64], D[64] of one step
  static constexpr int kOffBar = kOffVec + 2 * kVecBytes;
  static constexpr int kLayout = kOffBar + 256;
  static constexpr int kSmemAlloc = kLayout + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(192, 1)
wide_dk_kernel(const __grid_constant__ CUtensorMap map_q64, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do64,
               const __grid_constant__ CUtensorMap map_out, const BwdParams p) {
  using C = WideDkCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  if ((base - raw) + C::kLayout > static_cast<uint32_t>(C::kSmemAlloc)) {
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  const uint32_t s_k = base + C::kOffK, s_v = base + C::kOffV;
  auto s_slot = [&](int i) { return base + C::kOffSlot + i * kWSubTile; };
  auto s_ds = [&](int i) { return base + C::kOffDs + i * kWDs; };
  auto s_vec = [&](int i) { return base + C::kOffVec + i * C::kVecBytes; };
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_kv_full = bars;
  auto bar_full = [&](int i) { return bars + 8u + 8u * i; };           // slots (up to 4)
  auto bar_empty = [&](int i) { return bars + 40u + 8u * i; };
  auto bar_vec_full = [&](int i) { return bars + 72u + 8u * i; };
  auto bar_vec_empty = [&](int i) { return bars + 88u + 8u * i; };
  auto bar_s_full = [&](int i) { return bars + 104u + 8u * i; };
  auto bar_dp_full = [&](int i) { return bars + 120u + 8u * i; };
  auto bar_ready = [&](int i) { return bars + 136u + 8u * i; };        // dS^T written
  const uint32_t bar_o_final = bars + 152, bar_stall = bars + 160;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 168);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 172);
  const uint32_t bar_k_tmem = bars + 176;                               // every row of K copied into TMEM
  // TMEM: dK accumulator | S^T | dP^T | K (A operand of S^T). One buffer each
  // for S^T and dP^T, whose next products follow the warps' dS^T: step s uses
  // barrier 0 at phase parity s & 1.
  constexpr uint32_t kColKT = 384;
  auto tb = [&](int) { return 0; };
  auto tp = [&](int s) { return static_cast<uint32_t>(s & 1); };
  auto col_s = [&](int) { return kWColS; };
  const uint32_t col_dp = kWColS + 64u;

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
  const int nq64 = p.NQP / kWSub;
  // first 64-query sub-tile that sees key tile jt (bottom-right causal)
  const int first_row = jt * kBN - p.causal_off;
  const int s0 = p.causal ? (first_row <= 0 ? 0 : min(nq64, first_row / kWSub)) : 0;
  const int per_head = nq64 - s0;
  const int nsteps = (jt < nkt) ? G * per_head : 0;
  auto step_head = [&](int s) { return b * p.Hq + hk * G + s / per_head; };
  auto step_sub = [&](int s) { return s0 + s % per_head; };
  // slot of step s's Q and dO
  auto q_slot = [&](int s) { return (2 * s + 2) & 3; };
  auto do_slot = [&](int s) { return (2 * s + 3) & 3; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_kv_full, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_vec_full(i), 1);
      mbar_init(bar_vec_empty(i), 128);
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_dp_full(i), 1);
      mbar_init(bar_ready(i), 128);
    }
    mbar_init(bar_o_final, 1);
    mbar_init(bar_stall, 1);
    mbar_init(bar_k_tmem, 128);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_q64);
      tma_prefetch_map(&map_do64);
      mbar_arrive_expect_tx(bar_kv_full, 2 * kWTile);
      for (int bx = 0; bx < kWD / 64; ++bx) {
        tma_load_3d(s_k + bx * kBoxBytes, &map_k, bar_kv_full, bx * 64, jt * kBN, bhkv);
        tma_load_3d(s_v + bx * kBoxBytes, &map_v, bar_kv_full, bx * 64, jt * kBN, bhkv);
      }
      // per-slot use counts give the parity of each empty wait
      int uses[4] = {0, 0, 0, 0};
      auto load = [&](const CUtensorMap* m, int slot, int row0, int bh) -> bool {
        // slots 0 and 1 take Q/dO only once every row of K is in TMEM
        if (slot < 2 && uses[slot] == 0 && !mbar_wait(bar_k_tmem, 0, abort_flag, deadline)) return false;
        if (!mbar_wait(bar_empty(slot), (uses[slot] & 1) ^ 1, abort_flag, deadline)) return false;
        ++uses[slot];
        mbar_arrive_expect_tx(bar_full(slot), kWSubTile);
        for (int bx = 0; bx < kWD / 64; ++bx)
          tma_load_3d(s_slot(slot) + bx * kWSubBox, m, bar_full(slot), bx * 64, row0, bh);
        return true;
      };
      for (int s = 0; s < nsteps; ++s) {
        const int bh = step_head(s), row0 = step_sub(s) * kWSub;
        if (!load(&map_q64, q_slot(s), row0, bh)) break;
        const int vb = s & 1;
        if (!mbar_wait(bar_vec_empty(vb), ((s >> 1) & 1) ^ 1, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_vec_full(vb), 2 * kWSub * 4);
        const size_t voff = static_cast<size_t>(bh) * p.NQP + row0;
        bulk_load(s_vec(vb), p.ws_lse2 + voff, kWSub * 4, bar_vec_full(vb));
        bulk_load(s_vec(vb) + kWSub * 4, p.ws_d + voff, kWSub * 4, bar_vec_full(vb));
        if (!load(&map_do64, do_slot(s), row0, bh)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int fulls[4] = {0, 0, 0, 0};     // phases of each slot's full barrier waited for so far
      auto wait_full = [&](int slot) -> bool {
        return mbar_wait(bar_full(slot), (fulls[slot]++) & 1, abort_flag, deadline);
      };
      bool ok = !p.test_stall || mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      ok = ok && (nsteps == 0 || (mbar_wait(bar_kv_full, 0, abort_flag, deadline) &&
                                  mbar_wait(bar_k_tmem, 0, abort_flag, deadline)));
      auto scores = [&](int s) {       // S^T_s = K Q_s^T, A = K from TMEM
        const uint32_t id = make_idesc(1, 128, kWSub, 0, 0);
        const uint64_t bd = smem_desc_sw128(s_slot(q_slot(s)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk) {
          const uint32_t kb = kk * 32;
          mma_bf16_ts(tbase + col_s(s), tbase + kColKT + kk * 8, desc_add(bd, (kb / 128) * kWSubBox + kb % 128), id,
                      kk > 0);
        }
        mma_commit(bar_s_full(tb(s)));
      };
      auto dp = [&](int s) {           // dP^T_s; dO_s's slot is then free
        issue_scores(tbase + col_dp, s_v, s_slot(do_slot(s)));
        mma_commit(bar_dp_full(tb(s)));
        mma_commit(bar_empty(do_slot(s)));
      };
      {
        // order: S^T_0, dP^T_0; per step s: [dS^T_s] dK_s (Q_s's slot free
        // after), [Q_{s+1}] S^T_{s+1}, [dO_{s+1}] dP^T_{s+1}. dO_{s+1} can only
        // load once dK_s has freed its slot; S^T_{s+1} runs meanwhile. (S^T two
        // steps ahead put a second such load, Q_{s+2} behind dP^T_{s+1}, on the
        // issuer's path in every step.)
        if (ok && nsteps > 0) {
          ok = wait_full(q_slot(0));
          if (ok) { tc_fence_after(); scores(0); }
          ok = ok && wait_full(do_slot(0));
          if (ok) { tc_fence_after(); dp(0); }
        }
        for (int s = 0; s < nsteps && ok; ++s) {
          if (!(ok = mbar_wait(bar_ready(tb(s)), tp(s), abort_flag, deadline))) break;
          tc_fence_after();
          issue_acc_ss(tbase + kWColAcc, s_ds(s & 1), s_slot(q_slot(s)), s > 0);
          mma_commit(bar_empty(q_slot(s)));
          if (s + 1 < nsteps) {
            // the S^T and dP^T buffers were last read by the warps for step s
            // (their dS^T_s came first); dS^T buffer (s+1)&1 by dK_{s-1}, issued
            // before these products
            if (!(ok = wait_full(q_slot(s + 1)))) break;
            tc_fence_after();
            scores(s + 1);
            if (!(ok = wait_full(do_slot(s + 1)))) break;
            tc_fence_after();
            dp(s + 1);
          }
        }
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ one thread per key row
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int key = jt * kBN + r;
    const bool key_pad = key >= p.Nk;
    const float sl2 = p.scale_log2;
    bool ok = true;
    if (nsteps > 0) {
      // this key row of K into TMEM as the A operand of S^T (128 columns of
      // bf16 pairs, the tile's 16-byte units in order); then slots 0 and 1 are free
      ok = mbar_wait(bar_kv_full, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
#pragma unroll
        for (int bx = 0; bx < kWD / 64; ++bx) {
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[4 * u]), "=r"(w[4 * u + 1]), "=r"(w[4 * u + 2]), "=r"(w[4 * u + 3])
                         : "r"(swz128(s_k + bx * kBoxBytes, r, u)));
          tmem_st_32x32b_x32(tbase + lane_off + kColKT + 32u * bx, w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_k_tmem);
      }
    }
    for (int s = 0; s < nsteps && ok; ++s) {
      const int sb = s & 1;
      const int q0 = step_sub(s) * kWSub;
      ok = mbar_wait(bar_s_full(tb(s)), tp(s), abort_flag, deadline) &&
           mbar_wait(bar_vec_full(sb), (s >> 1) & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* vec = reinterpret_cast<const float*>(gbase + (s_vec(sb) - base));
      float x[64];
      tmem_ld64(tbase + lane_off + col_s(s), x);
      // P^T[key, q] = 2^(S^T s log2e - LSE_q log2e); causal: q + (Nk - N) >= key
      const int lim = key - p.causal_off - q0;             // first visible query column
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float e = ex2_approx(fmaf(x[c], sl2, -vec[c]));
        x[c] = (key_pad || (p.causal && c < lim)) ? 0.f : e;
      }
      {
        // dP^T_s only now: it may still wait for dO_s's load while P^T is formed
        ok = mbar_wait(bar_dp_full(tb(s)), tp(s), abort_flag, deadline);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float dpv[64];
        tmem_ld64(tbase + lane_off + col_dp, dpv);
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = x[c] * (dpv[c] - vec[kWSub + c]);
        // dS^T buffer sb was last read by dK_{s-2}, which completed before S^T_s
        store_row64(s_ds(sb), r, x);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_ready(tb(s)));
      }
      mbar_arrive(bar_vec_empty(sb));
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
        stage_acc_row(tbase + lane_off + kWColAcc, stg, r, p.scale);
      } else {
#pragma unroll
        for (int bx = 0; bx < kWD / 64; ++bx)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" :: "r"(swz128(stg + bx * kBoxBytes, r, u)), "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (!*abort_flag && warp == 2 && lane == 0 && jt < nkt) {
      for (int bx = 0; bx < kWD / 64; ++bx) tma_store_3d(&map_out, stg + bx * kBoxBytes, bx * 64, jt * kBN, bhkv);
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
// Shared memory: K | Q | dO (one [128, 256] bf16 tile each) | LSE x2 | barriers.
// TMEM: dV accumulator | S^T buffer 0 | S^T buffer 1 (128 columns each).
// With 128 queries per step S^T = K Q^T is an N = 128 product (an N = 64
// product takes about as long); Q and dO have one buffer each, so step t+1's
// Q loads once S^T_t has read step t's.
struct WideDvCfg {
  static constexpr int kOffK = 0;
  static constexpr int kOffQ = kWTile;
  static constexpr int kOffDo = 2 * kWTile;
  static constexpr int kOffVec = 3 * kWTile;
  static constexpr int kVecBytes = 512;                // LSE log2(e) of 128 queries
  static constexpr int kOffBar = kOffVec + 2 * kVecBytes;
  static constexpr int kLayout = kOffBar + 256;
  static constexpr int kSmemAlloc = kLayout + 1024;
  static constexpr uint32_t kColS = 256;               // buffers at 256 and 384
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(192, 1)
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
  const uint32_t s_k = base + C::kOffK, s_q = base + C::kOffQ, s_do = base + C::kOffDo;
  auto s_vec = [&](int i) { return base + C::kOffVec + i * C::kVecBytes; };
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_k_full = bars, bar_q_full = bars + 8, bar_q_empty = bars + 16;
  const uint32_t bar_do_full = bars + 24, bar_do_empty = bars + 32;
  auto bar_vec_full = [&](int i) { return bars + 40u + 8u * i; };
  auto bar_vec_empty = [&](int i) { return bars + 56u + 8u * i; };
  auto bar_s_full = [&](int i) { return bars + 72u + 8u * i; };
  auto bar_ready = [&](int i) { return bars + 88u + 8u * i; };      // P^T written over S^T
  const uint32_t bar_o_final = bars + 104, bar_stall = bars + 112;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 120);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 124);

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
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_empty, 1);
    mbar_init(bar_do_full, 1);
    mbar_init(bar_do_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_vec_full(i), 1);
      mbar_init(bar_vec_empty(i), 128);
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_ready(i), 128);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_do);
      mbar_arrive_expect_tx(bar_k_full, kWTile);
      for (int bx = 0; bx < kWD / 64; ++bx)
        tma_load_3d(s_k + bx * kBoxBytes, &map_k, bar_k_full, bx * 64, jt * kBN, bhkv);
      for (int t = 0; t < nsteps; ++t) {
        const int bh = step_head(t), it = step_tile(t);
        const uint32_t par = (t & 1) ^ 1;                // one buffer: phase t - 1 released it
        if (!mbar_wait(bar_q_empty, par, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_q_full, kWTile);
        for (int bx = 0; bx < kWD / 64; ++bx)
          tma_load_3d(s_q + bx * kBoxBytes, &map_q, bar_q_full, bx * 64, it * kBM, bh);
        const int vb = t & 1;
        if (!mbar_wait(bar_vec_empty(vb), ((t >> 1) & 1) ^ 1, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_vec_full(vb), C::kVecBytes);
        bulk_load(s_vec(vb), p.ws_lse2 + static_cast<size_t>(bh) * p.NQP + static_cast<size_t>(it) * kBM, C::kVecBytes,
                  bar_vec_full(vb));
        if (!mbar_wait(bar_do_empty, par, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_do_full, kWTile);
        for (int bx = 0; bx < kWD / 64; ++bx)
          tma_load_3d(s_do + bx * kBoxBytes, &map_do, bar_do_full, bx * 64, it * kBM, bh);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // S^T_0; per step t: [Q_{t+1} landed] S^T_{t+1} into the other buffer
    // (its P^T_{t-1} was read by dV_{t-1}, issued before), then [P^T_t
    // written, dO_t landed] dV_t. Each S^T frees Q's buffer once it completes,
    // each dV frees dO's.
    if (lane == 0) {
      bool ok = !p.test_stall || mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      ok = ok && (nsteps == 0 || mbar_wait(bar_k_full, 0, abort_flag, deadline));
      const uint32_t id_s = make_idesc(1, 128, 128, 0, 0);     // S^T: K and Q both K-major
      const uint32_t id_v = make_idesc(1, 128, kWD, 0, 1);     // dV: A = P^T from TMEM, B = dO MN-major
      const uint64_t kd = smem_desc_sw128(s_k, 16, 1024), qd = smem_desc_sw128(s_q, 16, 1024);
      const uint64_t dod = smem_desc_sw128(s_do, kBoxBytes, 1024);
      auto scores = [&](int t) {
        const uint32_t d = tbase + C::kColS + 128u * (t & 1);
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(d, desc_add(kd, off), desc_add(qd, off), id_s, kk > 0);
        }
        mma_commit(bar_s_full(t & 1));
        mma_commit(bar_q_empty);
      };
      if (ok && nsteps > 0) {
        ok = mbar_wait(bar_q_full, 0, abort_flag, deadline);
        if (ok) {
          tc_fence_after();
          scores(0);
        }
      }
      for (int t = 0; t < nsteps && ok; ++t) {
        if (t + 1 < nsteps) {
          if (!(ok = mbar_wait(bar_q_full, (t + 1) & 1, abort_flag, deadline))) break;
          tc_fence_after();
          scores(t + 1);
        }
        if (!(ok = mbar_wait(bar_ready(t & 1), (t >> 1) & 1, abort_flag, deadline))) break;
        if (!(ok = mbar_wait(bar_do_full, t & 1, abort_flag, deadline))) break;
        tc_fence_after();
        // dV += P^T dO (K = 128 queries; P^T of queries 2c, 2c+1 in column c of the buffer)
        const uint32_t a = tbase + C::kColS + 128u * (t & 1);
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          mma_bf16_ts(tbase + kWColAcc, a + kk * 8, desc_add(dod, kk * 16 * 128), id_v, t > 0 || kk > 0);
        mma_commit(bar_do_empty);
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ one thread per key row
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int key = jt * kBN + r;
    const bool key_pad = key >= p.Nk;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < nsteps && ok; ++t) {
      const int sb = t & 1;
      ok = mbar_wait(bar_s_full(sb), (t >> 1) & 1, abort_flag, deadline) &&
           mbar_wait(bar_vec_full(sb), (t >> 1) & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(gbase + (s_vec(sb) - base));
      const uint32_t ts = tbase + lane_off + C::kColS + 128u * sb;
      uint32_t sr[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld_32x32b_x32(ts + 32 * q4, sr[q4]);
      tmem_wait_ld();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) reg_fence_x32(sr[q4]);
      // P^T[key, q] = 2^(S^T s log2e - LSE_q log2e); causal: q + (Nk - N) >= key;
      // query rows past N have LSE = +inf, so P = 0
      const int lim = key - p.causal_off - step_tile(t) * kBM;   // first visible query column
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pp[32];
#pragma unroll
        for (int c2 = 0; c2 < 32; ++c2) {
          float e[2];
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int c = 64 * h + 2 * c2 + e2;
            const float pe = ex2_approx(fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, -lse2[c]));
            e[e2] = (key_pad || (p.causal && c < lim)) ? 0.f : pe;
          }
          pp[c2] = pack_bf16x2(e[0], e[1]);
        }
        // P^T over the S^T columns this thread has read: queries 64h + 2c2, +1 in column 32h + c2
        tmem_st_32x32b_x32(ts + 32 * h, pp);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_ready(sb));
      mbar_arrive(bar_vec_empty(sb));
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
        stage_acc_row(tbase + lane_off + kWColAcc, s_k, r, 1.0f);
      } else {
#pragma unroll
        for (int bx = 0; bx < kWD / 64; ++bx)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" :: "r"(swz128(s_k + bx * kBoxBytes, r, u)), "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (!*abort_flag && warp == 2 && lane == 0) {
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

// ------------------------------------------------------------------ dQ per query tile
// Shared memory: dO | four 32 KB slots | dS x2 | barriers. Q lands in slots
// 0 and 1, the warps copy it into TMEM as the A operand of S, and the slots
// then join a ring in which K_j and V_j are items 2j and 2j+1 in slot
// (item + 2) % 4. K_j is read by S_j and dQ_j, V_j only by dP_j.
struct WideDqCfg {
  static constexpr int kSlots = 4;
  static constexpr int kOffDo = 0;
  static constexpr int kOffSlot = kWTile;              // slots 0-1 first hold the Q tile
  static constexpr int kOffDs = kOffSlot + kSlots * kWSubTile;
  static constexpr int kOffBar = kOffDs + 2 * kWDs;
  // TMEM: dQ accumulator | S | dP | Q as the A operand of S (two bf16 per column)
  static constexpr uint32_t kColS = 256, kColDP = 320, kColQ = 384;
  static constexpr int kLayout = kOffBar + 256;
  static constexpr int kSmemAlloc = kLayout + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(192, 1)
wide_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k64,
               const __grid_constant__ CUtensorMap map_v64, const __grid_constant__ CUtensorMap map_do,
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
  auto s_slot = [&](int i) { return base + C::kOffSlot + i * kWSubTile; };
  const uint32_t s_q = s_slot(0);                      // the Q tile, then the dQ staging
  auto s_ds = [&](int i) { return base + C::kOffDs + i * kWDs; };
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_q_full = bars;                    // Q and dO landed
  auto bar_full = [&](int i) { return bars + 8u + 8u * i; };     // slots 0..3
  auto bar_empty = [&](int i) { return bars + 40u + 8u * i; };
  const uint32_t bar_s_full = bars + 72, bar_dp_full = bars + 80, bar_ready = bars + 88;
  const uint32_t bar_o_final = bars + 96, bar_stall = bars + 104;
  const uint32_t bar_q_tmem = bars + 112;              // every row of Q copied into TMEM
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 120);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 124);

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
  const int nk64 = (p.Nk + kWSub - 1) / kWSub;
  int nsteps = nk64;
  if (p.causal) {
    const int last = qt * kBM + kBM - 1 + p.causal_off;   // the tile's last row sees keys up to here
    nsteps = last < 0 ? 0 : min(nk64, last / kWSub + 1);
  }
  // ring of four slots: K_j and V_j are items 2j and 2j+1, in slot (item + 2) % 4,
  // so the first two go to slots 2 and 3 while Q still occupies slots 0 and 1
  auto k_slot = [&](int j) { return (2 * j + 2) & 3; };
  auto v_slot = [&](int j) { return (2 * j + 3) & 3; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_q_full, 1);
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(bar_full(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_ready, 128);
    mbar_init(bar_q_tmem, 128);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nsteps > 0) {
      tma_prefetch_map(&map_k64);
      tma_prefetch_map(&map_v64);
      mbar_arrive_expect_tx(bar_q_full, 2 * kWTile);
      for (int bx = 0; bx < kWD / 64; ++bx) {
        tma_load_3d(s_q + bx * kBoxBytes, &map_q, bar_q_full, bx * 64, qt * kBM, bh);
        tma_load_3d(s_do + bx * kBoxBytes, &map_do, bar_q_full, bx * 64, qt * kBM, bh);
      }
      int uses[C::kSlots] = {0, 0, 0, 0};
      auto load = [&](const CUtensorMap* m, int slot, int row0) -> bool {
        // slots 0 and 1 take K/V only once every row of Q is in TMEM
        if (slot < 2 && uses[slot] == 0 && !mbar_wait(bar_q_tmem, 0, abort_flag, deadline)) return false;
        if (!mbar_wait(bar_empty(slot), (uses[slot] & 1) ^ 1, abort_flag, deadline)) return false;
        ++uses[slot];
        mbar_arrive_expect_tx(bar_full(slot), kWSubTile);
        for (int bx = 0; bx < kWD / 64; ++bx)
          tma_load_3d(s_slot(slot) + bx * kWSubBox, m, bar_full(slot), bx * 64, row0, bh_kv);
        return true;
      };
      for (int j = 0; j < nsteps; ++j) {
        if (!load(&map_k64, k_slot(j), j * kWSub)) break;
        if (!load(&map_v64, v_slot(j), j * kWSub)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int fulls[C::kSlots] = {0, 0, 0, 0};
      auto wait_full = [&](int slot) -> bool {
        return mbar_wait(bar_full(slot), (fulls[slot]++) & 1, abort_flag, deadline);
      };
      bool ok = !p.test_stall || mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      ok = ok && (nsteps == 0 || (mbar_wait(bar_q_full, 0, abort_flag, deadline) &&
                                  mbar_wait(bar_q_tmem, 0, abort_flag, deadline)));
      auto scores = [&](int j) {     // S_j = Q K_j^T with Q from TMEM
        const uint32_t id = make_idesc(1, 128, kWSub, 0, 0);
        const uint64_t bd = smem_desc_sw128(s_slot(k_slot(j)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kWD / 16; ++kk) {
          const uint32_t kb = kk * 32;
          mma_bf16_ts(tbase + C::kColS, tbase + C::kColQ + kk * 8, desc_add(bd, (kb / 128) * kWSubBox + kb % 128), id,
                      kk > 0);
        }
        mma_commit(bar_s_full);
      };
      auto dp = [&](int j) {
        issue_scores(tbase + C::kColDP, s_do, s_slot(v_slot(j)));
        mma_commit(bar_dp_full);
        mma_commit(bar_empty(v_slot(j)));
      };
      // order: S_0, dP_0; per step j: [dS_j] dQ_j (K_j's slot free after),
      // [K_{j+1}] S_{j+1}, [V_{j+1}] dP_{j+1}. S and dP have one TMEM buffer
      // each: step j+1's are issued only after the warps' read of step j's
      // (the dS_j they waited for). With four slots K_{j+2} and V_{j+2} load
      // while step j+1 runs.
      if (ok && nsteps > 0) {
        ok = wait_full(k_slot(0));
        if (ok) { tc_fence_after(); scores(0); }
        ok = ok && wait_full(v_slot(0));
        if (ok) { tc_fence_after(); dp(0); }
      }
      for (int j = 0; j < nsteps && ok; ++j) {
        if (!(ok = mbar_wait(bar_ready, j & 1, abort_flag, deadline))) break;
        tc_fence_after();
        issue_acc_ss(tbase + kWColAcc, s_ds(j & 1), s_slot(k_slot(j)), j > 0);
        mma_commit(bar_empty(k_slot(j)));
        if (j + 1 < nsteps) {
          // dS buffer (j+1)&1 was last read by dQ_{j-1}, issued before these products
          if (!(ok = wait_full(k_slot(j + 1)))) break;
          tc_fence_after();
          scores(j + 1);
          if (!(ok = wait_full(v_slot(j + 1)))) break;
          tc_fence_after();
          dp(j + 1);
        }
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ one thread per query row
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int q = qt * kBM + r;
    const float sl2 = p.scale_log2;
    // this row's LSE log2(e) (+inf past N: P = 0) and D
    const float lse2 = p.ws_lse2[static_cast<size_t>(bh) * p.NQP + qt * kBM + r];
    const float dsub = p.ws_d[static_cast<size_t>(bh) * p.NQP + qt * kBM + r];
    const int key_lim = p.causal ? min(p.Nk, q + p.causal_off + 1) : p.Nk;   // keys < key_lim are visible
    bool ok = true;
    if (nsteps > 0) {
      // this row of Q into TMEM as the A operand of S: 128 columns of bf16
      // pairs, the lower dimension in the low half (the tile's 16-byte units
      // in order), then slots 0 and 1 are free for K and V
      ok = mbar_wait(bar_q_full, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
#pragma unroll
        for (int bx = 0; bx < kWD / 64; ++bx) {
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
      const int sb = j & 1;
      // P from S first: dP_j may still wait for V_j's load
      ok = mbar_wait(bar_s_full, j & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float x[64], dpv[64];
      tmem_ld64(tbase + lane_off + C::kColS, x);
      const int lim = key_lim - j * kWSub;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float pe = ex2_approx(fmaf(x[c], sl2, -lse2));
        x[c] = (c < lim) ? pe : 0.f;
      }
      ok = mbar_wait(bar_dp_full, j & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      tmem_ld64(tbase + lane_off + C::kColDP, dpv);
#pragma unroll
      for (int c = 0; c < 64; ++c) x[c] = x[c] * (dpv[c] - dsub);
      // dS buffer sb was last read by dQ_{j-2}, which completed before S_j
      store_row64(s_ds(sb), r, x);
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
        stage_acc_row(tbase + lane_off + kWColAcc, s_q, r, p.scale);
      } else {
#pragma unroll
        for (int bx = 0; bx < kWD / 64; ++bx)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" :: "r"(swz128(s_q + bx * kBoxBytes, r, u)), "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 128);
    if (!*abort_flag && warp == 2 && lane == 0) {
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
  wide_dk_kernel<<<kv_grid, kWThreads, WideDkCfg::kSmemAlloc, stream>>>(m64.q, m.k, m.v, m64.dO, m.dk, pk);
  r = cudaGetLastError();
  if (r != cudaSuccess) return r;
  wide_dq_kernel<<<q_grid, kWThreads, WideDqCfg::kSmemAlloc, stream>>>(m.q, m64.k, m64.v, m.dO, m.dq, pq);
  return cudaGetLastError();
}

}  // namespace fa
