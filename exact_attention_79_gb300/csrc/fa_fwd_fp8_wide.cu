// FP8 (e4m3) forward with one 128-row query tile per CTA, for head dimensions
// above 128 (multiples of 16 up to 256, all in the D = 256 kernel, the columns
// past d zero-filled): the inputs of
// fa_fwd_fp8.cu's quantisers (Q, K with one scale per 64-row block, V
// transposed with one scale per column), the same arithmetic (logits scaled
// per row and key block, a running max that may trail by 2^4, 2^4 P rounded to
// e4m3 for P V, V's scales applied to the output columns).
//
// Method: "Flash Attention V3技术解析" sections 1.3 and 3.2 (FP8 operands with
// the contracted dimension contiguous, block-wise scales);
// "4.3 FlashAttention-2与FlashAttention-3演进", FlashAttention-3 section 2;
// head dimensions up to 256: "Flash Attention-2", section
// "Снижение накладных расходов".
//
// 384 threads:
//   warps 0-7   softmax: two warps per TMEM lane quarter, one per 64-key half
//               of each 128-key tile, so each thread of a row pair works on 64
//               logits; the two halves agree on the row max through a shared-
//               memory exchange guarded by an mbarrier (bounded wait) and keep
//               separate partial row sums, added once at the end
//   warp 8      TMA producer: Q once, then K_j and V^T_j tiles into a ring of
//               slots (one tile each), in the order the tensor core consumes them
//   warp 9      tensor-core issuer (one thread)
//   warp 10     ring watcher: folds "V_j landed" into the P-ready barrier of
//               step j, observing every load in ring order; warp 11 idle
// An e4m3 row of D codes is D/128 boxes of 128 bytes: Q, a K tile ([128 keys x
// D]) and a V^T tile ([D rows x 128 keys], boxes at y = 0 and 128 adjacent, so
// one K-major descriptor with N = D spans them) take D x 128 bytes each. TMEM:
// O in columns [0, D), S buffers at 256 and 384; P (four codes per column)
// overwrites S as the A operand of P V. Tensor-core order: S_0, S_1, then per
// key tile j: P_j V_j, S_{j+2}. At e4m3 rate a key tile's tensor work (512
// cycles at D = 128, 1024 at D = 256) is short against the softmax of 128
// logits per row, which one warp per scheduler runs as one long dependent
// sequence; two warps per row quarter halve it and let the schedulers
// interleave them. The bf16 output tile (D x 256 bytes) is staged in ring
// slots 0-1, idle once the last P V has completed.
// The layout works for D = 128 as well, but there it measured slower than the
// two-tile kernel of fa_fwd_fp8.cu (0.205 against 0.182 ms at N = 8192, 16
// heads, causal: half the tensor work per key tile, the same softmax), so
// only D = 256 is instantiated. Splitting each row's softmax over two warps
// gained 2.5% over one warp per row (0.2335 against 0.2396 ms).
#include <algorithm>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

template <int D>
struct W8Cfg {
  static_assert(D == 128 || D == 256, "FP8 one-tile head dimensions");
  static constexpr int kBoxes = D / 128;                     // 128-byte boxes along d
  static constexpr int kTile = kBoxes * kBoxBytes;           // Q, a K tile or a V^T tile
  static constexpr int kSlots = 6 * 32768 / kTile;           // 6 (D = 256) or 12 (D = 128)
  // softmax warps 0-7 (two per row), then producer 8, issuer 9, watcher 10,
  // idle 11; the softmax warpgroups take registers from the last one
  // (setmaxnreg) and come first, as the schedulers favour lower warp indices
  static constexpr int kThreads = 384;
  static constexpr uint32_t kRegsSoftmax = 184, kRegsOther = 120;
  static_assert(256 * kRegsSoftmax + 128 * kRegsOther <= 384 * 168, "register split");
  static constexpr int kBarBytes = 384;
  static constexpr int kXchgBytes = 2 * 2 * 128 * 4;         // [step parity][half][row] fp32
  static constexpr int kLayout = kTile + kSlots * kTile + kBarBytes + kXchgBytes;
  static constexpr int kSmemAlloc = std::min(227 * 1024, kLayout + 1024);
  static_assert(kLayout + 512 <= kSmemAlloc, "shared memory budget");
  static_assert(2 * kTile == D * 128 * 2, "the bf16 O tile takes two ring slots");
};
constexpr int kW8RowBlock = 64;             // rows per Q / K scale

// Consumption order of the ring: K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
__device__ __forceinline__ int w8_item_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int w8_item_v(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(384, 1)
fwd_fp8_wide_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_vt, const __grid_constant__ CUtensorMap map_o,
                    const FwdParams p) {
  using C = W8Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  if ((base - raw) + C::kLayout > static_cast<uint32_t>(C::kSmemAlloc)) {
    // the layout needs the dynamic window within a few hundred bytes of a
    // 1 KB boundary; refuse (and report) rather than overrun
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t s_q = base;
  const uint32_t s_ring = base + C::kTile;
  const uint32_t bars = s_ring + C::kSlots * C::kTile;
  const uint32_t xbuf = bars + C::kBarBytes;
  auto slot_addr = [&](int s) { return s_ring + static_cast<uint32_t>(s) * C::kTile; };
  auto bar_full = [&](int s) { return bars + 8u * s; };                     // up to 12
  auto bar_empty = [&](int s) { return bars + 96u + 8u * s; };              // up to 12
  const uint32_t bar_q_full = bars + 192;
  auto bar_s_full = [&](int i) { return bars + 200u + 8u * i; };            // 2
  // P-ready of step j is barrier j % 2 (a warp holding S_{j+1} early must not
  // arrive for step j+1 inside step j's phase)
  auto bar_p_ready = [&](int j) { return bars + 216u + 8u * (j & 1); };
  const uint32_t bar_pv_done = bars + 232;
  const uint32_t bar_o_final = bars + 240;
  const uint32_t bar_stall = bars + 248;                                    // nothing arrives (timeout test)
  // row-max exchange of lane quarter q at step j: barrier (q, j % 2), 64 arrivals
  auto bar_xchg = [&](int q, int j) { return bars + 256u + 16u * q + 8u * (j & 1); };
  uint8_t* const gbars = gbase + (bars - base);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbars + 320);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbars + 324);
  auto xchg_addr = [&](int j, int half, int row) {
    return xbuf + static_cast<uint32_t>((((j & 1) * 2 + half) * 128 + row) * 4);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (query tile, batch*head); heads in L2-sized groups, the
  // heaviest causal tiles first inside a group
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
    const int last = qt * kBM + kBM - 1 + p.causal_off;     // bottom-right: key <= row + Nk - N
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
    mbar_init(bar_p_ready(0), 257);                 // 256 softmax threads + the watcher
    mbar_init(bar_p_ready(1), 257);
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_o_final, 1);
    mbar_init(bar_stall, 1);
    for (int q = 0; q < 4; ++q) {
      mbar_init(bar_xchg(q, 0), 64);
      mbar_init(bar_xchg(q, 1), 64);
    }
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
    setmaxnreg_dec<C::kRegsOther>();
    if (lane == 0 && n > 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_vt);
      mbar_arrive_expect_tx(bar_q_full, C::kTile);
      for (int bx = 0; bx < C::kBoxes; ++bx)
        tma_load_3d(s_q + bx * kBoxBytes, &map_q, bar_q_full, bx * 128, qt * kBM, bh);
      for (int it = 0; it < 2 * n; ++it) {
        bool is_v;
        int j;
        if (it == 0) { is_v = false; j = 0; }
        else if ((it & 1) && it <= 2 * n - 3) { is_v = false; j = (it + 1) >> 1; }
        else if (it & 1) { is_v = true; j = n - 1; }
        else { is_v = true; j = (it >> 1) - 1; }
        const int slot = it % C::kSlots;
        if (!mbar_wait(bar_empty(slot), ((it / C::kSlots) & 1u) ^ 1u, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_full(slot), C::kTile);
        const uint32_t dst = slot_addr(slot);
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          if (is_v)   // V^T rows [128 bx, 128 bx + 128) of d, the tile's 128 keys
            tma_load_3d(dst + bx * kBoxBytes, &map_vt, bar_full(slot), j * kBN, bx * 128, bh_kv);
          else        // K: the tile's 128 keys, columns [128 bx, 128 bx + 128) of d
            tma_load_3d(dst + bx * kBoxBytes, &map_k, bar_full(slot), bx * 128, j * kBN, bh_kv);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ tensor-core issuer
    setmaxnreg_dec<C::kRegsOther>();
    if (lane == 0 && n > 0) {
      const uint32_t idesc_qk = make_idesc(0, 128, 128, 0, 0);     // e4m3, both K-major
      const uint32_t idesc_pv = make_idesc(0, 128, D, 0, 0);       // A = P (TMEM), B = V^T K-major, N = D
      const uint64_t qdesc = smem_desc_sw128(s_q, 16, 1024);
      bool ok = true;
      if (p.test_stall) ok = mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      if (ok) ok = mbar_wait(bar_q_full, 0, abort_flag, deadline);
      // S_j = Q K_j^T into S buffer j % 2; the issuer waits for K_j itself
      auto issue_s = [&](int j) -> bool {
        const int it = w8_item_k(j);
        const int slot = it % C::kSlots;
        if (!mbar_wait(bar_full(slot), (it / C::kSlots) & 1, abort_flag, deadline)) return false;
        tc_fence_after();
        const uint64_t kd = smem_desc_sw128(slot_addr(slot), 16, 1024);
        const uint32_t d_tmem = tbase + 256u + 128u * (j & 1);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
          const uint32_t off = (kk / 4) * kBoxBytes + (kk % 4) * 32;   // 32 codes of d per step
          mma_fp8_ss(d_tmem, desc_add(qdesc, off), desc_add(kd, off), idesc_qk, kk > 0);
        }
        mma_commit(bar_s_full(j & 1));
        mma_commit(bar_empty(slot));
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int j = 0; j < n && ok; ++j) {
        // P_j written and V_j resident (folded in by the watcher)
        ok = mbar_wait(bar_p_ready(j), (j >> 1) & 1, abort_flag, deadline);
        if (!ok) break;
        tc_fence_after();
        const int vslot = w8_item_v(j, n) % C::kSlots;
        // O += P_j V_j: 32 keys per step, N = D across the boxes of V^T
        const uint64_t vd = smem_desc_sw128(slot_addr(vslot), 16, 1024);
        const uint32_t p_tmem = tbase + 256u + 128u * (j & 1);
#pragma unroll
        for (int kk = 0; kk < kBN / 32; ++kk)
          mma_fp8_ts(tbase, p_tmem + kk * 8, desc_add(vd, kk * 32), idesc_pv, j > 0 || kk > 0);
        mma_commit(bar_empty(vslot));
        mma_commit(bar_pv_done);
        // S_{j+2} overwrites P_j: issued after the P V that reads it
        if (j + 2 < n) ok = issue_s(j + 2);
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ------------------------------------------------------------ ring watcher
    setmaxnreg_dec<C::kRegsOther>();
    // Parity waits only tell phase k from phase k-1: every load is observed in
    // ring order, K loads only after the step's arrival (their latency never
    // holds P V back); a phase is arrived for only once its previous phase on
    // the same barrier has completed.
    if (warp == 10 && lane == 0 && n > 0) {
      auto landed = [&](int it) {
        return mbar_wait(bar_full(it % C::kSlots), (it / C::kSlots) & 1, abort_flag, deadline);
      };
      bool ok = landed(w8_item_k(0));
      if (ok && n > 1) ok = landed(w8_item_k(1));
      for (int j = 0; j < n && ok; ++j) {
        ok = landed(w8_item_v(j, n));
        if (ok && j >= 2) ok = mbar_wait(bar_p_ready(j), ((j >> 1) - 1) & 1, abort_flag, deadline);
        if (ok) mbar_arrive(bar_p_ready(j));
        if (ok && j + 2 < n) ok = landed(w8_item_k(j + 2));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    setmaxnreg_inc<C::kRegsSoftmax>();
    const int half = warp >> 2;                    // keys [64 half, 64 half + 64) of each tile
    const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_o = tbase + lane_off;
    const int q_row = qt * kBM + row;
    const int nqb = (p.N + kW8RowBlock - 1) / kW8RowBlock;
    const int nkb = (p.Nk + kW8RowBlock - 1) / kW8RowBlock;
    const float sq = p.q_scale[static_cast<size_t>(bh) * nqb + min(q_row / kW8RowBlock, nqb - 1)];
    const float* ksc = p.k_scale + static_cast<size_t>(bh_kv) * nkb;
    const float csq = p.scale_log2 * sq;
    float m = -INFINITY;                           // running max (up to 2^4 stale), log2 units; equal in both halves
    float l = 0.f;                                 // this half's running sum of 2^4 P
    bool ok = n > 0;
    for (int j = 0; j < n && ok; ++j) {
      const uint32_t t_s = tbase + lane_off + 256u + 128u * (j & 1);
      ok = mbar_wait(bar_s_full(j & 1), (j >> 1) & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld_32x32b_x32(t_s + 64 * half, sr[0]);
      tmem_ld_32x32b_x32(t_s + 64 * half + 32, sr[1]);
      tmem_wait_ld();
      reg_fence_x32(sr[0]);
      reg_fence_x32(sr[1]);
      float s[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      const int kv0 = j * kBN;
      int lim = kBN;
      if (p.causal) lim = min(lim, q_row + p.causal_off - kv0 + 1);
      if (kv0 + kBN > p.Nk) lim = min(lim, p.Nk - kv0);
      lim -= 64 * half;                            // limit within this half
      if (lim < 64) {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      // this half's multiplier: scale * log2(e) * sq * sk (its 64 keys are one K scale block)
      const float cm = csq * ksc[min(2 * j + half, nkb - 1)];
      float mk[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float* v = s + 32 * k;
        float a = fmax3(v[0], v[1], v[2]);
#pragma unroll
        for (int e = 3; e < 31; e += 2) a = fmax3(a, v[e], v[e + 1]);
        mk[k] = fmaxf(a, v[31]);
      }
      const float mine = fmaxf(mk[0], mk[1]) * cm;
      // exchange with the other half of the row (the buffer of step parity
      // j % 2 is rewritten at step j+2, after the partner's step-(j+1)
      // arrival, which follows its read below)
      st_shared_f32(xchg_addr(j, half, row), mine);
      mbar_arrive(bar_xchg(quarter, j));
      bool w = mbar_wait(bar_xchg(quarter, j), (j >> 1) & 1, abort_flag, deadline);
      w = __all_sync(0xffffffffu, w);
      if (!w) { ok = false; break; }
      const float other = ld_shared_f32(xchg_addr(j, half ^ 1, row));
      const float mx = half == 0 ? fmaxf(mine, other) : fmaxf(other, mine);
      const bool grow = mx > m + 4.0f;             // also true on the first tile (m = -inf)
      const float m_new = grow ? mx : m;
      const float alpha = grow ? ex2_approx(m - m_new) : 1.0f;
      m = m_new;
      const float off = (m == -INFINITY) ? 0.f : 4.0f - m;     // 2^4 P <= 256
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pr[16];
#pragma unroll
      for (int w4 = 0; w4 < 16; ++w4) {
        float x0, x1, x2, x3;
        fma2_bc(x0, x1, s[4 * w4], s[4 * w4 + 1], cm, off);
        fma2_bc(x2, x3, s[4 * w4 + 2], s[4 * w4 + 3], cm, off);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        add2_acc(sum0, sum1, p0, p1);
        add2_acc(sum0, sum1, p2, p3);
        pr[w4] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
      }
      tmem_st_32x32b_x16(t_s + 16 * half, pr);
      l = l * alpha + (sum0 + sum1);
      // O <- alpha O before P_j V_j, this half's columns: P_{j-1} V_{j-1} may
      // still be running (only P_{j-2} V_{j-2} precedes S_j), so wait for it;
      // phases up to j-2 have completed and phase j cannot before this
      // thread's P_j
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        bool wt = mbar_wait(bar_pv_done, (j - 1) & 1, abort_flag, deadline);
        wt = __all_sync(0xffffffffu, wt);
        if (!wt) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 2; cc += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + half * (D / 2) + cc, o);
          tmem_wait_ld();
          reg_fence_x32(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x32(t_o + half * (D / 2) + cc, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p_ready(j));
    }
    // ---------------------------------------------------------- epilogue
    const bool empty = n == 0;
    if (ok) {
      ok = mbar_wait(bar_o_final, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    // every softmax thread reaches the three barriers below, whatever its
    // waits returned; after the first, no loop step reads the exchange buffer
    named_bar_sync(1, 256);
    st_shared_f32(xchg_addr(0, half, row), l);
    named_bar_sync(1, 256);
    const float l_row = l + ld_shared_f32(xchg_addr(0, half ^ 1, row));
    if (ok || empty) {
      tc_fence_after();
      const float inv_l = l_row > 0.f ? 1.0f / l_row : 0.f;
      const float* vsc = p.v_scale + static_cast<size_t>(bh_kv) * p.head_dim;
      auto vscale = [&](int c) { return c < p.head_dim ? __ldg(vsc + c) : 0.f; };
      // bf16 O (128 x D, boxes of 64 columns) staged in ring slots 0-1: every
      // load has been consumed and the last P V has completed. This half
      // stages columns [half D/2, half D/2 + D/2).
      const uint32_t stage = s_ring;
#pragma unroll
      for (int c0 = half * (D / 2); c0 < half * (D / 2) + D / 2; c0 += 32) {
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
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 8 * u + 2 * e;
            wv[e] = pack_bf16x2(__uint_as_float(o[c]) * (vscale(c0 + c) * inv_l),
                                __uint_as_float(o[c + 1]) * (vscale(c0 + c + 1) * inv_l));
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, row, u0 + u)),
                       "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3]) : "memory");
        }
      }
      fence_proxy_async_smem();
      if (half == 0 && q_row < p.N)
        p.lse[static_cast<size_t>(bh) * p.N + q_row] = l_row > 0.f ? (m + log2f(l_row) - 4.0f) * kLn2 : -INFINITY;
    }
    named_bar_sync(1, 256);
    if (!*abort_flag && warp == 0 && lane == 0) {
      // 64-column boxes; one that would start at or past d is skipped
      for (int bx = 0; bx < D / 64; ++bx)
        if (bx * 64 < p.head_dim) tma_store_3d(&map_o, s_ring + bx * kBoxBytes, bx * 64, qt * kBM, bh);
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

template <int D>
static cudaError_t launch_w8(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mvt,
                             const CUtensorMap& mo, FwdParams p, cudaStream_t stream) {
  using C = W8Cfg<D>;
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    return cudaFuncSetAttribute(fwd_fp8_wide_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  });
  if (e != cudaSuccess) return e;
  // heads per group: their K and V^T codes (2 Nk D bytes per query head) within 64 MB
  const long long kv_bytes = 2LL * p.Nk * D;
  p.head_group = static_cast<int>(std::max(1LL, std::min<long long>(p.BH, (64LL << 20) / kv_bytes)));
  const long long grid = static_cast<long long>((p.N + kBM - 1) / kBM) * p.BH;
  fwd_fp8_wide_kernel<D><<<static_cast<unsigned>(grid), C::kThreads, C::kSmemAlloc, stream>>>(mq, mk, mvt, mo, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8_wide(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mvt,
                                const CUtensorMap& mo, FwdParams p, cudaStream_t stream) {
  if (p.head_dim <= 128 || p.head_dim > 256) return cudaErrorInvalidValue;
  return launch_w8<256>(mq, mk, mvt, mo, p, stream);
}

}  // namespace fa
