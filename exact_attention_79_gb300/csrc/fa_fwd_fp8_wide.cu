// FP8 (e4m3) forward for head dimensions 192 and 256 on sm_103a: the inputs
// of fa_fwd_fp8.cu's quantisers (Q, K with one scale per 64-row block, V
// transposed with one scale per column), the arithmetic of its attention
// kernel (logits scaled per row and key block, a running max that may trail by
// 2^4, 2^4 P rounded to e4m3 for P V, V's scales applied to the output
// columns), laid out like the wide-head bf16 forward.
//
// Method: "Flash Attention V3技术解析" sections 1.3 and 3.2 (FP8 operands with
// the contracted dimension contiguous, block-wise scales);
// "4.3 FlashAttention-2与FlashAttention-3演进", FlashAttention-3 section 2;
// head dimensions up to 256: "Flash Attention-2", section
// "Снижение накладных расходов".
//
// One CTA owns one 128-row query tile, 224 threads:
//   warp 0     TMA producer: Q once, then K_j and V^T_j tiles into a ring of
//              six 32 KB slots, in the order the tensor core consumes them
//   warp 1     tensor-core issuer (one thread) + TMEM owner
//   warps 2-5  softmax, one thread per query row
//   warp 6     ring watcher: folds "V_j landed" into the P-ready barrier of
//              step j, observing every load in ring order
// An e4m3 row of d = 256 is 256 bytes, so Q, a K tile ([128 keys x 256]) and
// a V^T tile ([256 d rows x 128 keys]) are two 128-byte-swizzled boxes each,
// 32 KB, one ring slot. TMEM: O in columns [0, 256), S buffers at 256 and 384;
// P (four codes per column) overwrites S as the A operand of P V. Tensor-core
// order: S_0, S_1, then per key tile j: P_j V_j, S_{j+2}. At e4m3 rate a key
// tile's tensor work (1024 cycles) sits below the softmax of one tile, so the
// second S buffer, which lets S_{j+1} be ready when the softmax gets to it,
// is what keeps the pipeline full. The bf16 output tile (64 KB) is staged in
// the ring, idle once the last P V has completed.
#include <algorithm>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {
namespace {

constexpr int kW8D = 256;                   // head dimension of the kernel (d = 192 runs in it, zero-filled)
constexpr int kW8Tile = 2 * kBoxBytes;      // 32 KB: Q, a K tile or a V^T tile
constexpr int kW8Slots = 6;
constexpr int kW8Threads = 224;
constexpr int kW8BarBytes = 256;
constexpr int kW8Smem = kW8Tile + kW8Slots * kW8Tile + kW8BarBytes + 1024;
static_assert(kW8Smem <= 227 * 1024, "shared memory budget");
constexpr int kW8RowBlock = 64;             // rows per Q / K scale

// Consumption order of the ring: K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
__device__ __forceinline__ int w8_item_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int w8_item_v(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

}  // namespace

__global__ void __launch_bounds__(224, 1)
fwd_fp8_wide_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_vt, const __grid_constant__ CUtensorMap map_o,
                    const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t s_q = base;
  const uint32_t s_ring = base + kW8Tile;
  const uint32_t bars = s_ring + kW8Slots * kW8Tile;
  auto slot_addr = [&](int s) { return s_ring + static_cast<uint32_t>(s) * kW8Tile; };
  auto bar_full = [&](int s) { return bars + 8u * s; };                     // kW8Slots
  auto bar_empty = [&](int s) { return bars + 48u + 8u * s; };              // kW8Slots
  const uint32_t bar_q_full = bars + 96;
  auto bar_s_full = [&](int i) { return bars + 104u + 8u * i; };            // 2
  // P-ready of step j is barrier j % 2 (a warp holding S_{j+1} early must not
  // arrive for step j+1 inside step j's phase)
  auto bar_p_ready = [&](int j) { return bars + 120u + 8u * (j & 1); };
  const uint32_t bar_pv_done = bars + 136;
  const uint32_t bar_o_final = bars + 144;
  const uint32_t bar_stall = bars + 152;                                    // nothing arrives (timeout test)
  uint8_t* const gbars = gbase + (bars - base);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbars + 160);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbars + 164);

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
    for (int s = 0; s < kW8Slots; ++s) {
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
    if (lane == 0 && n > 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_vt);
      mbar_arrive_expect_tx(bar_q_full, kW8Tile);
      for (int bx = 0; bx < 2; ++bx) tma_load_3d(s_q + bx * kBoxBytes, &map_q, bar_q_full, bx * 128, qt * kBM, bh);
      for (int it = 0; it < 2 * n; ++it) {
        bool is_v;
        int j;
        if (it == 0) { is_v = false; j = 0; }
        else if ((it & 1) && it <= 2 * n - 3) { is_v = false; j = (it + 1) >> 1; }
        else if (it & 1) { is_v = true; j = n - 1; }
        else { is_v = true; j = (it >> 1) - 1; }
        const int slot = it % kW8Slots;
        if (!mbar_wait(bar_empty(slot), ((it / kW8Slots) & 1u) ^ 1u, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_full(slot), kW8Tile);
        const uint32_t dst = slot_addr(slot);
        for (int bx = 0; bx < 2; ++bx) {
          if (is_v)   // V^T rows [128 bx, 128 bx + 128) of d, the tile's 128 keys
            tma_load_3d(dst + bx * kBoxBytes, &map_vt, bar_full(slot), j * kBN, bx * 128, bh_kv);
          else        // K: the tile's 128 keys, columns [128 bx, 128 bx + 128) of d
            tma_load_3d(dst + bx * kBoxBytes, &map_k, bar_full(slot), bx * 128, j * kBN, bh_kv);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ tensor-core issuer
    if (lane == 0 && n > 0) {
      const uint32_t idesc_qk = make_idesc(0, 128, 128, 0, 0);     // e4m3, both K-major
      const uint32_t idesc_pv = make_idesc(0, 128, kW8D, 0, 0);    // A = P (TMEM), B = V^T K-major, N = 256
      const uint64_t qdesc = smem_desc_sw128(s_q, 16, 1024);
      bool ok = true;
      if (p.test_stall) ok = mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      if (ok) ok = mbar_wait(bar_q_full, 0, abort_flag, deadline);
      // S_j = Q K_j^T into S buffer j % 2; the issuer waits for K_j itself
      auto issue_s = [&](int j) -> bool {
        const int it = w8_item_k(j);
        const int slot = it % kW8Slots;
        if (!mbar_wait(bar_full(slot), (it / kW8Slots) & 1, abort_flag, deadline)) return false;
        tc_fence_after();
        const uint64_t kd = smem_desc_sw128(slot_addr(slot), 16, 1024);
        const uint32_t d_tmem = tbase + 256u + 128u * (j & 1);
#pragma unroll
        for (int kk = 0; kk < kW8D / 32; ++kk) {
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
        const int vslot = w8_item_v(j, n) % kW8Slots;
        // O += P_j V_j: 32 keys per step, N = 256 across both 128-row boxes of V^T
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
  } else if (warp == 6) {
    // ------------------------------------------------------------ ring watcher
    // Parity waits only tell phase k from phase k-1: every load is observed in
    // ring order, K loads only after the step's arrival (their latency never
    // holds P V back); a phase is arrived for only once its previous phase on
    // the same barrier has completed.
    if (lane == 0 && n > 0) {
      auto landed = [&](int it) {
        return mbar_wait(bar_full(it % kW8Slots), (it / kW8Slots) & 1, abort_flag, deadline);
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
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_o = tbase + lane_off;
    const int q_row = qt * kBM + row;
    const int nqb = (p.N + kW8RowBlock - 1) / kW8RowBlock;
    const int nkb = (p.Nk + kW8RowBlock - 1) / kW8RowBlock;
    const float sq = p.q_scale[static_cast<size_t>(bh) * nqb + min(q_row / kW8RowBlock, nqb - 1)];
    const float* ksc = p.k_scale + static_cast<size_t>(bh_kv) * nkb;
    const float csq = p.scale_log2 * sq;
    float m = -INFINITY;                           // running max (up to 2^4 stale), log2 units
    float l = 0.f;                                 // running sum of 2^4 P
    bool ok = n > 0;
    for (int j = 0; j < n && ok; ++j) {
      const uint32_t t_s = tbase + lane_off + 256u + 128u * (j & 1);
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
      const int kv0 = j * kBN;
      int lim = kBN;
      if (p.causal) lim = min(lim, q_row + p.causal_off - kv0 + 1);
      if (kv0 + kBN > p.Nk) lim = min(lim, p.Nk - kv0);
      if (lim < kBN) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
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
      const float off = (m == -INFINITY) ? 0.f : 4.0f - m;     // 2^4 P <= 256
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pr[32];
#pragma unroll
      for (int w = 0; w < 32; ++w) {
        const float cm = (w < 16) ? c0 : c1;
        float x0, x1, x2, x3;
        fma2_bc(x0, x1, s[4 * w], s[4 * w + 1], cm, off);
        fma2_bc(x2, x3, s[4 * w + 2], s[4 * w + 3], cm, off);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        add2_acc(sum0, sum1, p0, p1);
        add2_acc(sum0, sum1, p2, p3);
        pr[w] = pack_e4m3x2(p0, p1) | (pack_e4m3x2(p2, p3) << 16);
      }
      tmem_st_32x32b_x32(t_s, pr);
      l = l * alpha + (sum0 + sum1);
      // O <- alpha O before P_j V_j: P_{j-1} V_{j-1} may still be running
      // (only P_{j-2} V_{j-2} precedes S_j), so wait for it; phases up to j-2
      // have completed and phase j cannot before this thread's P_j
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        bool w = mbar_wait(bar_pv_done, (j - 1) & 1, abort_flag, deadline);
        w = __all_sync(0xffffffffu, w);
        if (!w) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kW8D; cc += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(t_o + cc, o);
          tmem_wait_ld();
          reg_fence_x32(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st_32x32b_x32(t_o + cc, o);
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
    if (ok || empty) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const float* vsc = p.v_scale + static_cast<size_t>(bh_kv) * p.head_dim;
      auto vscale = [&](int c) { return c < p.head_dim ? __ldg(vsc + c) : 0.f; };
      // bf16 O (128 x 256, four boxes of 64 columns) staged in the ring: every
      // load has been consumed and the last P V has completed
      const uint32_t stage = s_ring;
#pragma unroll
      for (int c0 = 0; c0 < kW8D; c0 += 32) {
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
      if (q_row < p.N)
        p.lse[static_cast<size_t>(bh) * p.N + q_row] = l > 0.f ? (m + log2f(l) - 4.0f) * kLn2 : -INFINITY;
    }
    named_bar_sync(1, 128);
    if (!*abort_flag && warp == 2 && lane == 0) {
      // 64-column boxes; one that would start at or past d is skipped
      for (int bx = 0; bx < 4; ++bx)
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

cudaError_t launch_fwd_fp8_wide(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mvt,
                                const CUtensorMap& mo, FwdParams p, cudaStream_t stream) {
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    return cudaFuncSetAttribute(fwd_fp8_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kW8Smem);
  });
  if (e != cudaSuccess) return e;
  // heads per group: their K and V^T codes (2 Nk d bytes per query head) within 64 MB
  const long long kv_bytes = 2LL * p.Nk * kW8D;
  p.head_group = static_cast<int>(std::max(1LL, std::min<long long>(p.BH, (64LL << 20) / kv_bytes)));
  const long long grid = static_cast<long long>((p.N + kBM - 1) / kBM) * p.BH;
  fwd_fp8_wide_kernel<<<static_cast<unsigned>(grid), kW8Threads, kW8Smem, stream>>>(mq, mk, mvt, mo, p);
  return cudaGetLastError();
}

}  // namespace fa
