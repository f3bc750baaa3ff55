// Forward exact attention on sm_103a with CTA pairs (tcgen05 cta_group::2),
// bf16, head dimension up to 128: the same method as fa_fwd.cu (tiled online
// softmax with a running max and sum, "FlashAttention技术解析" 2.1-2.2; the
// division by l deferred to the end, "FlashAttention v2相比于v1有哪些更新"
// section 3; ping-pong of two softmax groups against one MMA-issuing thread,
// "Flash Attention V3技术解析" 1.2; causal blocks above the diagonal skipped,
// same page 2.1), laid out for two SMs at once.
//
// One cluster of two CTAs covers four 128-row query tiles of one (batch,
// head): CTA r holds tiles A = 4p + r and B = 4p + 2 + r. One thread of the
// even CTA issues every MMA as an M = 256 product over both CTAs:
//   S_A = [Q_A(cta 0); Q_A(cta 1)] K_j^T     N = 128 keys, K = d
//   O_A += [P_A(cta 0); P_A(cta 1)] V_j      N = d, K = 128 keys
// and likewise for B. A pair MMA reads half of B from each CTA (split along
// N), so each CTA loads only its half of every key/value tile: keys
// [64 r, 64 r + 64) of K_j and columns [64 r, 64 r + 64) of V_j. Against two
// independent CTAs this halves the MMA instructions, commits and polls per
// unit of work and the K/V bytes each SM loads (the ring holds twice as many
// tiles). It does not lower the rate at which the one issuing thread must
// start MMAs: an M = 256 product keeps both SMs busy for the time an M = 128
// product keeps one busy. Each hand-off also gains a step across the cluster
// and waits for the slower of eight warps. Measured on GB300 it is slower than
// the one-CTA kernel (fa_fwd.cu) and gives the same bits, so it is reached
// only through fa_fwd_pair.
//
// Roles (352 threads per CTA):
//   warp 0      TMA producer (both CTAs): Q tiles, then K / V halves into a ring
//   warp 1      TMEM allocation (both CTAs, collectively); the MMA issuer (even CTA)
//   warps 2-5   softmax group 0 (tile A), one thread per query row (both CTAs)
//   warps 6-9   softmax group 1 (tile B)
//   warp 10     even CTA: ring watcher (operands landed -> P-ready, slots back to
//               both producers); odd CTA: forwarder (its Q and K_0 landed -> one
//               remote arrival; its V_j and K_{j+1} landed -> one remote arrival
//               on the even CTA's P-ready barrier of step j)
// The odd CTA's softmax warps arrive on the even CTA's P-ready barriers
// directly (one remote arrival per warp), so the issuer waits on one barrier
// per group and step for both CTAs.
// TMEM per CTA (512 columns): S_A | S_B | O_A | O_B, each CTA its own 128 rows.
// Both tiles of a pair run the same key-tile range: the longer of the two
// (the tile below it in the causal order sees one fully masked key tile).
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kPD = 128;                            // head-dimension build
constexpr int kPTile = kPD / 64 * kBoxBytes;        // one [128, d] bf16 tile: 32 KB
constexpr int kPHalf = kPTile / 2;                  // one ring item: half a K or V tile, 16 KB
constexpr int kPStages = 10;
constexpr int kPBarBytes = 512;
constexpr int kPSmem = 2 * kPTile + kPStages * kPHalf + kPBarBytes + 1024;
constexpr int kPThreads = 352;
static_assert(kPSmem <= 227 * 1024, "shared memory budget");

}  // namespace

__global__ void __launch_bounds__(352, 1)
fwd_pair_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k64,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const uint32_t s_q[2] = {base, base + kPTile};
  const uint32_t s_kv = base + 2 * kPTile;
  const uint32_t bars = s_kv + kPStages * kPHalf;
  auto bar_q_full = [&](int i) { return bars + 8u * i; };
  auto bar_kv_full = [&](int s) { return bars + 16u + 8u * s; };
  auto bar_kv_empty = [&](int s) { return bars + 16u + 8u * (kPStages + s); };
  auto bar_s_full = [&](int i) { return bars + 16u + 16u * kPStages + 8u * i; };
  auto bar_p_ready = [&](int i) { return bars + 32u + 16u * kPStages + 8u * i; };
  auto bar_o_final = [&](int i) { return bars + 48u + 16u * kPStages + 8u * i; };
  const uint32_t bar_peer_start = bars + 64u + 16u * kPStages;    // even CTA: the odd CTA's Q and K_0 landed
  const uint32_t bar_stall = bars + 72u + 16u * kPStages;         // nothing arrives (timeout test)
  uint8_t* const gbars = gbase + (bars - base);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbars + 80 + 16 * kPStages);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbars + 84 + 16 * kPStages);
  unsigned long long* const clock_start = reinterpret_cast<unsigned long long*>(gbars + 96 + 16 * kPStages);  // [2]
  static_assert(112 + 16 * kPStages <= kPBarBytes, "barrier area");

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(blockIdx.x & 1);       // == %cluster_ctarank for clusters of two
  const bool leader = rank == 0;
  const uint32_t peer = static_cast<uint32_t>(rank ^ 1);

  // ---- work item: (cluster of four query tiles, batch * head), heaviest first
  const int lin = static_cast<int>(blockIdx.x >> 1);
  const int quad = p.num_pairs - 1 - lin / p.BH;
  const int bh = lin % p.BH;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int bh_kv = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int nq = (p.N + kBM - 1) / kBM;
  const int nk = (p.Nk + kBN - 1) / kBN;
  const int qt[2] = {4 * quad + rank, 4 * quad + 2 + rank};
  auto reach = [&](int t) {
    if (!p.causal) return nk;
    const int last = t * kBM + kBM - 1 + p.causal_off;
    return last < 0 ? 0 : min(nk, last / kBN + 1);
  };
  // key tiles of group g: the longer range of the pair's two tiles (tiles past
  // the last query tile count as absent); identical in both CTAs
  auto group_steps = [&](int g) {
    const int t0 = 4 * quad + 2 * g, t1 = t0 + 1;
    const int a = t0 < nq ? reach(t0) : 0, c = t1 < nq ? reach(t1) : 0;
    return a > c ? a : c;
  };
  const int nkv[2] = {group_steps(0), group_steps(1)};
  const int nmax = nkv[0] > nkv[1] ? nkv[0] : nkv[1];

  if (threadIdx.x == 0) {
    clock_mark(clock_start);
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_q_full(i), 1);
      mbar_init(bar_s_full(i), 1);
      // even CTA: its 128 threads, its watcher, the odd CTA's 4 warps and forwarder
      mbar_init(bar_p_ready(i), 134);
      mbar_init(bar_o_final(i), 1);
    }
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_peer_start, 1);
    mbar_init(bar_stall, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();        // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint64_t deadline = global_timer_ns() + p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k64);
      tma_prefetch_map(&map_v);
      for (int i = 0; i < 2; ++i) {
        if (nkv[i] == 0) continue;
        // a tile past N reads as zeros and is never stored; its rows still
        // take part in the pair's MMAs
        mbar_arrive_expect_tx(bar_q_full(i), kPTile);
        for (int bx = 0; bx < kPD / 64; ++bx)
          tma_load_3d(s_q[i] + bx * kBoxBytes, &map_q, bar_q_full(i), bx * 64, qt[i] * kBM, bh);
      }
      for (int c = 0; c < 2 * nmax; ++c) {
        const int slot = c % kPStages;
        const uint32_t round = c / kPStages;
        // slots come back from the even CTA's watcher (a remote arrival here)
        if (!mbar_wait_cluster(bar_kv_empty(slot), (round & 1u) ^ 1u, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_kv_full(slot), kPHalf);
        const uint32_t dst = s_kv + slot * kPHalf;
        const int j = c >> 1;
        if ((c & 1) == 0) {
          // K_j, keys [64 r, 64 r + 64): d / 64 boxes of 64 rows
          for (int bx = 0; bx < kPD / 64; ++bx)
            tma_load_3d(dst + bx * (kBoxBytes / 2), &map_k64, bar_kv_full(slot), bx * 64, j * kBN + 64 * rank, bh_kv);
        } else {
          // V_j, columns [64 r, 64 r + 64): one box of 128 keys
          tma_load_3d(dst, &map_v, bar_kv_full(slot), 64 * rank, j * kBN, bh_kv);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (leader && lane == 0) {
      const uint32_t idesc_qk = make_idesc(1, 256, 128, 0, 0);
      const uint32_t idesc_pv = make_idesc(1, 256, kPD, 0, 1);
      bool ok = true;
      if (p.test_stall) ok = mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      for (int i = 0; i < 2 && ok; ++i)
        if (nkv[i] > 0) ok = mbar_wait(bar_q_full(i), 0, abort_flag, deadline);
      if (ok && nmax > 0) ok = mbar_wait(bar_kv_full(0), 0, abort_flag, deadline) &&
                               mbar_wait_cluster(bar_peer_start, 0, abort_flag, deadline);
      int c = 0;
      auto issue_qk = [&](int i, uint32_t sk) {
        const uint64_t qd = smem_desc_sw128(s_q[i], 16, 1024), kd = smem_desc_sw128(sk, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kPD / 16; ++kk) {
          const uint32_t kb = kk * 32;               // byte offset along d
          mma_bf16_ss_pair(tbase + 128u * i, desc_add(qd, (kb / 128) * kBoxBytes + kb % 128),
                           desc_add(kd, (kb / 128) * (kBoxBytes / 2) + kb % 128), idesc_qk, kk > 0);
        }
      };
      auto issue_pv = [&](int i, uint32_t sv, bool acc) {
        // V half: 128 keys x 64 columns, MN-major; 16 keys per MMA
        const uint64_t vd = smem_desc_sw128(sv, kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16_ts_pair(tbase + 256u + kPD * i, tbase + 128u * i + kk * 8, desc_add(vd, kk * 16 * 128), idesc_pv,
                           acc || kk > 0);
      };
      if (ok && nmax > 0) {
        tc_fence_after();
        const uint32_t sk = s_kv;                    // K_0: load 0, slot 0
        ++c;
        for (int i = 0; i < 2; ++i) {
          if (nkv[i] == 0) continue;
          issue_qk(i, sk);
          mma_commit_pair(bar_s_full(i), 3);
        }
      }
      for (int j = 0; j < nmax && ok; ++j) {
        // residency of V_j and K_{j+1} in both CTAs is folded into the P-ready barriers
        const uint32_t sv = s_kv + (c % kPStages) * kPHalf;
        ++c;
        uint32_t sk_next = 0;
        if (j + 1 < nmax) {
          sk_next = s_kv + (c % kPStages) * kPHalf;
          ++c;
        }
        for (int i = 0; i < 2; ++i) {
          if (j >= nkv[i]) continue;
          if (!mbar_wait_cluster(bar_p_ready(i), j & 1, abort_flag, deadline)) { ok = false; break; }
          tc_fence_after();
          issue_pv(i, sv, j > 0);
          if (j + 1 < nkv[i]) {
            issue_qk(i, sk_next);
            mma_commit_pair(bar_s_full(i), 3);
          } else {
            mma_commit_pair(bar_o_final(i), 3);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp >= 10) {
    if (leader && lane == 0) {
      // -------------------------------------------------------- ring watcher (even CTA)
      const int L = (nkv[1] == nmax) ? 1 : 0;        // the group whose S MMAs go last in each step
      // parity waits only tell phase k from phase k-1: observe every phase of
      // every slot in order, starting with K_0
      bool ok = nmax == 0 || mbar_wait(bar_kv_full(0), 0, abort_flag, deadline);
      auto hand_p = [&](int i, int j) {
        if (j > 0) ok = mbar_wait_cluster(bar_p_ready(i), (j - 1) & 1, abort_flag, deadline);
        if (ok) mbar_arrive(bar_p_ready(i));
      };
      auto release = [&](int slot) {
        mbar_arrive(bar_kv_empty(slot));
        // relaxed: the MMAs that read the slot have completed (S_L(j) observed)
        mbar_arrive_remote_relaxed(mapa_shared(bar_kv_empty(slot), peer));
      };
      for (int j = 0; j < nmax && ok; ++j) {
        const int cv = 2 * j + 1;
        ok = mbar_wait(bar_kv_full(cv % kPStages), (cv / kPStages) & 1, abort_flag, deadline);
        if (ok && j + 1 < nmax) {
          const int ck = 2 * j + 2;
          ok = mbar_wait(bar_kv_full(ck % kPStages), (ck / kPStages) & 1, abort_flag, deadline);
        }
        if (ok && L == 1 && j < nkv[0]) hand_p(0, j);
        // S_L(j) done: issued after every MMA that reads K_j or V_{j-1}, in both CTAs
        if (ok) ok = mbar_wait(bar_s_full(L), j & 1, abort_flag, deadline);
        if (ok) {
          release((2 * j) % kPStages);
          if (j > 0) release((2 * j - 1) % kPStages);
        }
        if (ok) hand_p(L, j);
      }
    } else if (!leader && lane == 0) {
      // -------------------------------------------------------- forwarder (odd CTA)
      bool ok = true;
      for (int i = 0; i < 2 && ok; ++i)
        if (nkv[i] > 0) ok = mbar_wait(bar_q_full(i), 0, abort_flag, deadline);
      if (ok && nmax > 0) ok = mbar_wait(bar_kv_full(0), 0, abort_flag, deadline);
      if (ok && nmax > 0) mbar_arrive_remote_relaxed(mapa_shared(bar_peer_start, peer));   // loads observed landed
      for (int j = 0; j < nmax && ok; ++j) {
        const int cv = 2 * j + 1;
        ok = mbar_wait(bar_kv_full(cv % kPStages), (cv / kPStages) & 1, abort_flag, deadline);
        if (ok && j + 1 < nmax) {
          const int ck = 2 * j + 2;
          ok = mbar_wait(bar_kv_full(ck % kPStages), (ck / kPStages) & 1, abort_flag, deadline);
        }
        for (int i = 0; i < 2 && ok; ++i) {
          if (j >= nkv[i]) continue;
          // S_i(j) done means the even CTA's P-ready(i) completed phase j - 1
          // (S_i(j) is issued after it), so this arrival counts for phase j
          ok = mbar_wait(bar_s_full(i), j & 1, abort_flag, deadline);
          if (ok) mbar_arrive_remote_relaxed(mapa_shared(bar_p_ready(i), peer));   // loads observed landed
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax groups (both CTAs)
    const int g = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int n_kv = nkv[g];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tbase + lane_off + 128u * g;
    const uint32_t t_o = tbase + lane_off + 256u + kPD * g;
    const int q_row = qt[g] * kBM + row;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;
    float l = 0.f;
    bool ok = n_kv > 0;
    const uint32_t p_ready_remote = mapa_shared(bar_p_ready(g), 0);
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
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
      // mask: causal (bottom-right), the ragged key tail; a row past its own
      // reach (the shorter tile of the pair) sees the whole tile masked
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
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
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
      // O <- alpha O before the next P V: the previous P V of this group has
      // completed (it was issued before the S MMA just waited for)
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c0 = 0; c0 < kPD; c0 += 32) {
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
      if (leader) {
        mbar_arrive(bar_p_ready(g));
      } else {
        __syncwarp();
        // for the warp's 32 rows; relaxed: tcgen05.wait::st above returned, so
        // P is in TMEM before the arrival, and the P V that reads it is issued
        // only after the phase completes (the release form cost 18% of the kernel)
        if (lane == 0) mbar_arrive_remote_relaxed(p_ready_remote);
      }
    }
    // ---------------------------------------------------------- epilogue
    const bool empty = n_kv == 0;
    if (ok) {
      ok = mbar_wait(bar_o_final(g), 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok || empty) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const uint32_t stage = s_q[g];     // Q tile no longer needed: all its MMAs completed
#pragma unroll
      for (int c0 = 0; c0 < kPD; c0 += 32) {
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
          for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[8 * u + 2 * e]) * inv_l, __uint_as_float(o[8 * u + 2 * e + 1]) * inv_l);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, row, u0 + u)),
                       "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
        }
      }
      fence_proxy_async_smem();
      if (q_row < p.N) p.lse[static_cast<size_t>(bh) * p.N + q_row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
    named_bar_sync(1 + g, 128);
    if (qt[g] < nq && !*abort_flag && warp == 2 + 4 * g && lane == 0) {
      for (int bx = 0; bx < kPD / 64; ++bx) tma_store_3d(&map_o, s_q[g] + bx * kBoxBytes, bx * 64, qt[g] * kBM, bh);
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
  // neither CTA leaves while the pair's MMAs or the other CTA's remote
  // arrivals may still touch its shared memory
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tbase, 512);
  if (threadIdx.x == 0) clock_record(p.clock_acc, clock_start);
}

cudaError_t launch_fwd_pair(const CUtensorMap& mq, const CUtensorMap& mk64, const CUtensorMap& mv,
                            const CUtensorMap& mo, FwdParams p, cudaStream_t stream) {
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    return cudaFuncSetAttribute(fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  });
  if (e != cudaSuccess) return e;
  const int nq = (p.N + kBM - 1) / kBM;
  p.num_pairs = (nq + 3) / 4;              // clusters (four query tiles) per head
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.num_pairs * p.BH);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_pair_kernel, mq, mk64, mv, mo, p);
}

}  // namespace fa
