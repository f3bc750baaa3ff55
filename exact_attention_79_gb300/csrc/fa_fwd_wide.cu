// Forward exact attention for head dimensions 136..256 on sm_103a: the same
// computation as fa_fwd.cu (online softmax over 128-key tiles, output divided
// by the running sum once at the end, natural-log logsumexp), laid out for
// operands twice as wide.
//
// Method: "FlashAttention技术解析" 2.1-2.2 (tiling, online softmax);
// "FlashAttention v2相比于v1有哪些更新" section 3 (deferred rescale, the
// logsumexp as the only saved statistic); "Flash Attention V3技术解析" 1.2
// (a producer warp feeding the tensor core through a shared-memory ring) and
// 2.1 (causal tiles above the diagonal skipped). Head dimensions up to 256:
// "Flash Attention-2", section "Снижение накладных расходов".
//
// Why a second kernel. At d = 256 one 128-row fp32 output accumulator takes
// 256 of the 512 TMEM columns and a 128 x 256 bf16 tile takes 64 KB of shared
// memory, so the two-query-tile layout of the d <= 128 kernel fits neither.
// Here one CTA owns one 128-row query tile:
//   warp 0     TMA producer: Q once, then K and V pieces into a ring of
//              32 KB slots, in the order the tensor core consumes them
//   warp 1     tensor-core issuer (one thread) + TMEM owner
//   warps 2-5  softmax, one thread per query row
//   warp 6     ring watcher: waits for V_j to land and adds one arrival to
//              the P-ready barrier of step j, so the issuing thread learns "P_j
//              written and V_j resident" from one barrier instead of three
//              (each poll costs it about as much as issuing two or three MMAs).
//              K_{j+2} it still waits for itself, just before S_{j+2}: folding
//              that load into P-ready too would hold P_j V_j back by the load
//              latency, which the ring's depth does not cover.
// The ring holds 160 KB against 128 KB of operands in use, so a load can only
// start about one MMA group before it is needed. The producer therefore also
// asks L2 for the pieces three items ahead (a prefetch needs no slot), which
// turns most ring loads into L2 hits.
// TMEM (512 columns x 128 lanes, fp32): O in columns [0, D), two S buffers at
// 256 and 384, so S_{j+1} is computed while the softmax works on S_j.
// Shared memory: Q [128 x D] (D/64 boxes of 128 rows x 128 bytes), then five
// 32 KB slots. A K tile is split along d into two pieces of at most two
// boxes (each S MMA step reads 16 columns of d from one box); a V tile is
// split along the keys into two 64-key halves of D/64 boxes of 64 rows x 128
// bytes (each P V MMA step reads 16 keys from one half). Splitting therefore
// adds no MMA instructions, and a deeper ring hides the TMA latency.
// Tensor-core order: S_0, S_1, then per key tile j: P_j V_j, S_{j+2}. The
// rescale of O (only when a row max grows by more than 2^8 in log2 units)
// waits for the previous P V to complete, which the issuer signals per tile.
#include <algorithm>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

template <int D>
struct WideCfg {
  static_assert(D == 192 || D == 256, "wide head dimensions");
  static constexpr int kNBox = D / 64;                    // 64-column boxes along d
  static constexpr int kQBytes = kNBox * kBoxBytes;       // Q tile (and the staged O tile)
  static constexpr int kSlotBytes = 32768;
  static constexpr int kVBoxBytes = 64 * 128;             // 64 keys x 128 bytes
  static constexpr int kSlots = 5;
  static constexpr int kThreads = 224;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 256;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = kQBytes + kSlots * kSlotBytes + kBarBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(D + 2 * 128 <= 512, "TMEM budget");
  // bytes of K piece `pc` (boxes 2pc, 2pc+1 when they exist) and of a V half
  __host__ __device__ static constexpr uint32_t k_piece_bytes(int pc) {
    return (kNBox - 2 * pc >= 2 ? 2 : 1) * kBoxBytes;
  }
  static constexpr uint32_t kVHalfBytes = kNBox * kVBoxBytes;
};

// Consumption order of the ring, in items of two slot loads each:
// K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
__device__ __forceinline__ int wide_item_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int wide_item_v(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

template <int D>
__global__ void __launch_bounds__(224, 1)
fwd_wide_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                const FwdParams p) {
  using C = WideCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t s_q = base;
  const uint32_t s_ring = base + C::kQBytes;
  const uint32_t bars = s_ring + C::kSlots * C::kSlotBytes;
  auto slot_addr = [&](int s) { return s_ring + static_cast<uint32_t>(s) * C::kSlotBytes; };
  auto bar_full = [&](int s) { return bars + 8u * s; };                     // kSlots
  auto bar_empty = [&](int s) { return bars + 40u + 8u * s; };              // kSlots
  const uint32_t bar_q_full = bars + 80;
  auto bar_s_full = [&](int i) { return bars + 88u + 8u * i; };             // 2
  // P-ready of step j is barrier j % 2. A softmax thread that has written P_j
  // may already hold S_{j+1} (issued a step earlier) and write P_{j+1} before
  // the slowest thread arrives for step j: with a single barrier that arrival
  // would count toward step j. S_{j+2} is issued only after step j's barrier
  // completes, so no thread gets two steps ahead on the same barrier.
  auto bar_p_ready = [&](int j) { return (j & 1) ? bars + 144u : bars + 104u; };
  const uint32_t bar_pv_done = bars + 112;
  const uint32_t bar_o_final = bars + 120;
  const uint32_t bar_stall = bars + 128;                                    // nothing arrives (timeout test)
  uint8_t* const gbars = gbase + (bars - base);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbars + 136);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbars + 140);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (query tile, batch*head). Heads go in groups of
  // p.head_group whose K and V fit in part of L2; inside a group the
  // heaviest causal tiles come first, so the last CTAs are light ones.
  const int lin = blockIdx.x;
  const int nq = (p.N + kBM - 1) / kBM;
  const int grp = lin / (nq * p.head_group);
  const int gsize = min(p.head_group, p.BH - grp * p.head_group);
  const int local = lin - grp * p.head_group * nq;
  const int qt = nq - 1 - local / gsize;
  const int bh = grp * p.head_group + local % gsize;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bh_kv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int nk = (p.Nk + kBN - 1) / kBN;
  int n = nk;
  if (p.causal) {
    // key tiles up to the one holding key (last row + Nk - N); none if negative
    const int last = qt * kBM + kBM - 1 + p.causal_off;
    n = last < 0 ? 0 : min(nk, last / kBN + 1);
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_q_full, 1);
    mbar_init(bar_s_full(0), 1);
    mbar_init(bar_s_full(1), 1);
    mbar_init(bar_p_ready(0), 129);                 // 128 softmax threads + the watcher
    mbar_init(bar_p_ready(1), 129);
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_o_final, 1);
    mbar_init(bar_stall, 1);
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
    if (lane == 0 && n > 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      mbar_arrive_expect_tx(bar_q_full, C::kQBytes);
      for (int bx = 0; bx < C::kNBox; ++bx)
        tma_load_3d(s_q + bx * kBoxBytes, &map_q, bar_q_full, bx * 64, qt * kBM, bh);
      bool ok = true;
      for (int it = 0; it < 2 * n && ok; ++it) {
        // item `it` of the consumption order: K_j or V_j
        bool is_v;
        int j;
        if (it == 0) { is_v = false; j = 0; }
        else if ((it & 1) && it <= 2 * n - 3) { is_v = false; j = (it + 1) >> 1; }
        else if (it & 1) { is_v = true; j = n - 1; }
        else { is_v = true; j = (it >> 1) - 1; }
        if (it + 3 < 2 * n) {
          // L2 prefetch of item it + 3 (the same decoding as below)
          const int it3 = it + 3;
          bool v3;
          int j3;
          if ((it3 & 1) && it3 <= 2 * n - 3) { v3 = false; j3 = (it3 + 1) >> 1; }
          else if (it3 & 1) { v3 = true; j3 = n - 1; }
          else { v3 = true; j3 = (it3 >> 1) - 1; }
          for (int bx = 0; bx < C::kNBox; ++bx) {
            if (v3) {
              tma_prefetch_l2_3d(&map_v, bx * 64, j3 * kBN, bh_kv);
              tma_prefetch_l2_3d(&map_v, bx * 64, j3 * kBN + 64, bh_kv);
            } else {
              tma_prefetch_l2_3d(&map_k, bx * 64, j3 * kBN, bh_kv);
            }
          }
        }
        for (int pc = 0; pc < 2 && ok; ++pc) {
          const int ld = 2 * it + pc;
          const int slot = ld % C::kSlots;
          ok = mbar_wait(bar_empty(slot), ((ld / C::kSlots) & 1u) ^ 1u, abort_flag, deadline);
          if (!ok) break;
          const uint32_t dst = slot_addr(slot);
          if (!is_v) {
            // K piece pc: columns [128 pc, 128 pc + 128) of d, all 128 keys
            mbar_arrive_expect_tx(bar_full(slot), C::k_piece_bytes(pc));
            for (int bx = 2 * pc; bx < 2 * pc + 2 && bx < C::kNBox; ++bx)
              tma_load_3d(dst + (bx - 2 * pc) * kBoxBytes, &map_k, bar_full(slot), bx * 64, j * kBN, bh_kv);
          } else {
            // V half pc: keys [64 pc, 64 pc + 64) of the tile, all of d
            mbar_arrive_expect_tx(bar_full(slot), C::kVHalfBytes);
            for (int bx = 0; bx < C::kNBox; ++bx)
              tma_load_3d(dst + bx * C::kVBoxBytes, &map_v, bar_full(slot), bx * 64, j * kBN + 64 * pc, bh_kv);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ tensor-core issuer
    if (lane == 0 && n > 0) {
      const uint32_t idesc_qk = make_idesc(1, 128, 128, 0, 0);
      const uint32_t idesc_pv = make_idesc(1, 128, D, 0, 1);
      const uint64_t qdesc = smem_desc_sw128(s_q, 16, 1024);
      bool ok = true;
      if (p.test_stall) ok = mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      if (ok) ok = mbar_wait(bar_q_full, 0, abort_flag, deadline);
      // the slots of item `it` (V residency comes folded into P-ready)
      auto take = [&](int it, int& s0, int& s1) {
        s0 = (2 * it) % C::kSlots;
        s1 = (2 * it + 1) % C::kSlots;
      };
      // S_j = Q K_j^T into S buffer j % 2. Each K piece is waited for just
      // before the MMAs that read it and handed back right after them, which
      // gives the second piece's load half an S product more time.
      auto issue_s = [&](int j) -> bool {
        const int it = wide_item_k(j);
        int s0, s1;
        take(it, s0, s1);
        const uint32_t d_tmem = tbase + C::kColS0 + 128u * (j & 1);
        const uint64_t kd0 = smem_desc_sw128(slot_addr(s0), 16, 1024);
        const uint64_t kd1 = smem_desc_sw128(slot_addr(s1), 16, 1024);
        if (!mbar_wait(bar_full(s0), ((2 * it) / C::kSlots) & 1, abort_flag, deadline)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int bx = kk / 4;                       // box along d
          const uint32_t in_box = (kk % 4) * 32;       // 16 columns = 32 bytes
          if (kk == 8) {
            mma_commit(bar_empty(s0));
            if (!mbar_wait(bar_full(s1), ((2 * it + 1) / C::kSlots) & 1, abort_flag, deadline)) return false;
            tc_fence_after();
          }
          const uint64_t kd = desc_add(bx < 2 ? kd0 : kd1, (bx & 1) * kBoxBytes + in_box);
          mma_bf16_ss(d_tmem, desc_add(qdesc, bx * kBoxBytes + in_box), kd, idesc_qk, kk > 0);
        }
        mma_commit(bar_s_full(j & 1));
        mma_commit(bar_empty(s1));
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int j = 0; j < n && ok; ++j) {
        // P_j written and V_j resident
        ok = mbar_wait(bar_p_ready(j), (j >> 1) & 1, abort_flag, deadline);
        int s0 = 0, s1 = 0;
        take(wide_item_v(j, n), s0, s1);
        if (!ok) break;
        tc_fence_after();
        // O += P_j V_j: A = P_j (bf16 pairs in the S buffer), B = V_j, MN-major
        const uint32_t p_tmem = tbase + C::kColS0 + 128u * (j & 1);
        const uint64_t vd0 = smem_desc_sw128(slot_addr(s0), C::kVBoxBytes, 1024);
        const uint64_t vd1 = smem_desc_sw128(slot_addr(s1), C::kVBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          mma_bf16_ts(tbase, p_tmem + kk * 8, desc_add(kk < 4 ? vd0 : vd1, (kk % 4) * 16 * 128), idesc_pv,
                      j > 0 || kk > 0);
          if (kk == 3) mma_commit(bar_empty(s0));    // first 64 keys read
        }
        mma_commit(bar_empty(s1));
        mma_commit(bar_pv_done);
        // S_{j+2} overwrites P_j: issued after the P V that reads it, and one
        // thread's MMAs complete in order
        if (j + 2 < n) ok = issue_s(j + 2);
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ ring watcher
    if (lane == 0 && n > 0) {
      // A parity wait only tells phase k from phase k-1, so a waiter must know
      // that the previous load into a slot has landed before it waits for the
      // next one. The watcher observes every load in ring order; it waits for
      // K_{j+2} only after its step-j arrival, so that load's latency never
      // holds P_j V_j back. The issuer waits for the K loads alone: the load
      // before one of them in the same slot was read by an MMA it issued after
      // P-ready or after its own wait, so it had landed.
      auto landed = [&](int it) -> bool {
        const int l0 = 2 * it, l1 = 2 * it + 1;
        return mbar_wait(bar_full(l0 % C::kSlots), (l0 / C::kSlots) & 1, abort_flag, deadline) &&
               mbar_wait(bar_full(l1 % C::kSlots), (l1 / C::kSlots) & 1, abort_flag, deadline);
      };
      bool ok = landed(wide_item_k(0));
      if (ok && n > 1) ok = landed(wide_item_k(1));
      for (int j = 0; j < n && ok; ++j) {
        ok = landed(wide_item_v(j, n));
        // arrive for step j only once step j-2 (the previous phase of the
        // same barrier) has completed
        if (ok && j >= 2) ok = mbar_wait(bar_p_ready(j), ((j >> 1) - 1) & 1, abort_flag, deadline);
        if (ok) mbar_arrive(bar_p_ready(j));
        if (ok && j + 2 < n) ok = landed(wide_item_k(j + 2));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;           // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_o = tbase + lane_off;
    const int q_row = qt * kBM + row;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;                           // running max, log2 units of scale*s
    float l = 0.f;                                 // running sum relative to m
    bool ok = n > 0;
    for (int j = 0; j < n && ok; ++j) {
      const uint32_t t_s = tbase + lane_off + C::kColS0 + 128u * (j & 1);
      ok = mbar_wait(bar_s_full(j & 1), (j >> 1) & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_ld_32x32b_x32(t_s + q4 * 32, sr[q4]);
      tmem_wait_ld();
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) reg_fence_x32(sr[q4]);
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

      // mask: causal (bottom-right: key <= row + Nk - N) and the ragged key tail
      int lim = kBN;
      const int kv0 = j * kBN;
      if (p.causal) lim = min(lim, q_row + p.causal_off - kv0 + 1);
      if (kv0 + kBN > p.Nk) lim = min(lim, p.Nk - kv0);
      if (lim < kBN) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      float mk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float* v = s + 32 * k;
        float a = fmax3(v[0], v[1], v[2]);
#pragma unroll
        for (int e = 3; e < 31; e += 2) a = fmax3(a, v[e], v[e + 1]);
        mk[k] = fmaxf(a, v[31]);
      }
      const float mx = fmax3(mk[0], mk[1], fmaxf(mk[2], mk[3])) * sl2;
      const bool grow = mx > m + 8.0f;             // also true on the first tile (m = -inf)
      const float m_new = grow ? mx : m;
      const float alpha = grow ? ex2_approx(m - m_new) : 1.0f;
      m = m_new;
      const float neg_m = (m == -INFINITY) ? 0.f : -m;   // a row with no visible key yet keeps P = 0
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t pr[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x0, x1;
          fma2_bc(x0, x1, s[h2 * 64 + 2 * c], s[h2 * 64 + 2 * c + 1], sl2, neg_m);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          add2_acc(sum0, sum1, p0, p1);
          pr[c] = pack_bf16x2(p0, p1);
        }
        tmem_st_32x32b_x32(t_s + h2 * 32, pr);
      }
      l = l * alpha + (sum0 + sum1);
      // O <- alpha O before P_j V_j accumulates: P_{j-1} V_{j-1} may still be
      // running (only P_{j-2} V_{j-2} precedes S_j), so wait for it. Phases of
      // that barrier up to j-2 have completed and phase j cannot complete
      // before this warp's P_j, so the parity wait is unambiguous.
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        bool w = mbar_wait(bar_pv_done, (j - 1) & 1, abort_flag, deadline);
        w = __all_sync(0xffffffffu, w);
        if (!w) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + c0, o);
          tmem_wait_ld();
          reg_fence_x32(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x32(t_o + c0, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p_ready(j));
    }
    // ---------------------------------------------------------- epilogue
    // A query tile that sees no key tile (more queries than keys under the
    // causal rule) skips the loop and writes O = 0, LSE = -inf; so does any
    // row that saw no key (l = 0).
    const bool empty = n == 0;
    if (ok) {
      ok = mbar_wait(bar_o_final, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok || empty) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      // the Q tile is free: every S MMA completed before the last P V
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        if (!empty) {
          tmem_ld_32x32b_x32(t_o + c0, o);
          tmem_wait_ld();
          reg_fence_x32(o);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0u;
        }
        const uint32_t box = s_q + (c0 / 64) * kBoxBytes;
        const int u0 = (c0 % 64) / 8;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[8 * u + 2 * e]) * inv_l, __uint_as_float(o[8 * u + 2 * e + 1]) * inv_l);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, row, u0 + u)),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
        }
      }
      fence_proxy_async_smem();
      if (q_row < p.N) p.lse[static_cast<size_t>(bh) * p.N + q_row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
    // all four warps meet here whether or not their waits succeeded; after a
    // timeout the abort flag is up and nothing is stored
    named_bar_sync(1, 128);
    if (!*abort_flag && warp == 2 && lane == 0) {
      for (int bx = 0; bx < C::kNBox; ++bx) tma_store_3d(&map_o, s_q + bx * kBoxBytes, bx * 64, qt * kBM, bh);
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

template <int D>
static cudaError_t launch_wide(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                               const CUtensorMap& mo, const FwdParams& p, cudaStream_t stream) {
  using C = WideCfg<D>;
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    return cudaFuncSetAttribute(fwd_wide_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>((p.N + kBM - 1) / kBM) * p.BH;
  // heads per group: their K and V (2 Nk D bf16 each, counted per query head)
  // within 64 MB, half of L2
  FwdParams q = p;
  const long long kv_bytes = 4LL * p.Nk * D;
  q.head_group = static_cast<int>(std::max(1LL, std::min<long long>(p.BH, (64LL << 20) / kv_bytes)));
  fwd_wide_kernel<D><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemBytes, stream>>>(mq, mk, mv, mo, q);
  return cudaGetLastError();
}

cudaError_t launch_fwd_wide(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mo, const FwdParams& p, cudaStream_t stream) {
  // d in (128, 192] runs in the 192 kernel and (192, 256] in the 256 one; the
  // last 64-column box is partly past d, read as zeros and clipped on store
  if (d > 128 && d <= 192) return launch_wide<192>(mq, mk, mv, mo, p, stream);
  if (d > 192 && d <= 256) return launch_wide<256>(mq, mk, mv, mo, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
