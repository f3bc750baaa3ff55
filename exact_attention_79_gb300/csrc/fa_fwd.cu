// Forward exact attention on sm_103a: O = softmax(scale Q K^T [+ causal]) V
// and the per-row natural-log logsumexp, with the N x N scores never leaving
// the SM.
//
// Method (pages on FlashAttention v1-v3):
//  * tiling over key/value blocks with an online softmax that keeps a running
//    max m and running sum l per query row ("FlashAttention技术解析" 2.1-2.2);
//  * output kept unnormalised, divided by l once at the end
//    ("FlashAttention v2相比于v1有哪些更新" section 3, "Rescale操作");
//  * Q outer, K/V inner, each CTA owns its output tile, no atomics in the
//    forward (same page, section 5; "FlashAttention技术解析" section 7);
//  * producer / consumer warp specialisation and ping-pong of two softmax
//    groups against the tensor core ("Flash Attention V3技术解析" 1.2);
//  * causal blocks above the diagonal skipped ("Flash Attention V3技术解析" 2.1).
//
// GB300 mapping. One CTA = two 128-row query tiles of one (batch, head).
// bf16 (384 threads, three warpgroups):
//   warps 0-3   softmax group 0 (query tile 0), one thread per query row
//   warps 4-7   softmax group 1 (query tile 1)
//   warp 8      TMA producer: Q tiles once, then K_j, V_j into a slot ring
//   warp 9      tensor-core issuer (one thread)
//   warp 10     ring watcher (below); warp 11 has no role
// The softmax warpgroups take registers from the last one (setmaxnreg): 184
// per thread against 120, where one register budget for all would be 168,
// at which the softmax spills. They come first: the schedulers favour lower
// warp indices, and with the watcher ahead of them the long-sequence forward
// ran 4-8% slower. fp32 (320 threads): warp 0 producer, warp 1 issuer, warps
// 2-5 the single tile's softmax.
//   ring watcher (bf16): waits for V_j and K_{j+1} to land and
//               adds one arrival to each group's P-ready barrier, so the
//               issuer learns "P_j written and its operands resident" from a
//               single barrier; it also hands ring slots back to the producer
//               once the last S MMA that follows their readers has completed.
//               Each barrier poll or commit of the issuing thread costs tens
//               to hundreds of cycles during which no MMA is queued, and the
//               issue queue holds only about three MMAs.
// TMEM (512 columns x 128 lanes, fp32): S0 | S1 | O0 | O1. The probabilities P
// overwrite S in place (bf16 pairs, or tf32) and feed O += P V with A read
// from TMEM. The rescale of O happens only when a row max grows by more than
// 2^8 (log2 units of the scaled logits); O and l always share the same
// reference max, so the final O / l and LSE are unchanged by that choice.
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

template <typename T, int D>
struct FwdCfg {
  static constexpr int kElt = sizeof(T);
  static constexpr bool kTf32 = (kElt == 4);
  static constexpr int kChunk = 128 / kElt;           // elements per 128-byte swizzle row
  static constexpr int kNBox = D / kChunk;            // TMA boxes per 128-row tile
  static constexpr int kTileBytes = kNBox * kBoxBytes;
  static constexpr int kUmmaK = 32 / kElt;            // K per MMA instruction (32 bytes)
  // K/V slot ring, as deep as shared memory allows: the next K tile is
  // loaded into the slot the producer got back two tiles ago, and a shallow
  // ring leaves its TMA latency exposed to the tensor core at every tile.
  static constexpr int kStages = kTf32 ? 3 : ((kTileBytes == 16384) ? 12 : 5);
  static constexpr int kThreads = kTf32 ? 320 : 384;      // bf16: softmax warpgroups 0-1, then producer, issuer, watcher, idle
  static constexpr int kSm0 = kTf32 ? 2 : 0;              // first softmax warp
  static constexpr int kProd = kTf32 ? 0 : 8, kIss = kTf32 ? 1 : 9;
  // bf16 register split (setmaxnreg): 256 softmax threads x 184 + 128 x 120 = 62464
  // of the 384 x 168 = 64512 the CTA is launched with
  static constexpr uint32_t kRegsSoftmax = 184, kRegsOther = 120;
  static_assert(kTf32 || 256 * kRegsSoftmax + 128 * kRegsOther <= 384 * 168, "register split");
  static constexpr uint32_t kTmemCols = 512;
  static __device__ __forceinline__ uint32_t col_s(int i) { return 128u * i; }
  static __device__ __forceinline__ uint32_t col_o(int i) { return 256u + D * i; }
  static constexpr int kBarBytes = 512;
  // fp32 extra buffers: the low tf32 parts of Q and of the current K tile
  static constexpr int kSmemBytes = (2 + kStages + (kTf32 ? 2 : 0)) * kTileBytes + kBarBytes + 1024;
  static constexpr uint32_t kFmt = kTf32 ? 2u : 1u;
  // tf32 operands must be K-major, so V (d contiguous) cannot feed the P V
  // product directly: the fp32 variant runs one query tile per CTA and its
  // softmax group transposes each V tile into a K-major V^T buffer (the idle
  // second query-tile slot). To keep the logits (and so the logsumexp) at
  // fp32 accuracy, Q and K are split into tf32 high and low parts and
  // S = Qhi Khi + Qhi Klo + Qlo Khi. bf16 runs two ping-ponged query tiles
  // per CTA.
  static constexpr bool kPingPong = !kTf32;
  static constexpr int kTilesPerCta = kPingPong ? 2 : 1;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(2 * 128 + 2 * D <= 512, "TMEM budget");
};

template <typename T, int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t sq, uint32_t sk, uint32_t idesc,
                                         uint32_t sq_lo = 0, uint32_t sk_lo = 0) {
  using C = FwdCfg<T, D>;
  const uint64_t qd = smem_desc_sw128(sq, 16, 1024), kd = smem_desc_sw128(sk, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / C::kUmmaK; ++kk) {
    const uint32_t kb = kk * 32;                              // byte offset along d
    const uint32_t off = (kb / 128) * kBoxBytes + (kb % 128);
    const uint64_t a = desc_add(qd, off);
    const uint64_t b = desc_add(kd, off);
    if constexpr (C::kTf32) {
      mma_tf32_ss(d_tmem, a, b, idesc, kk > 0);
      mma_tf32_ss(d_tmem, a, smem_desc_sw128(sk_lo + off, 16, 1024), idesc, 1);
      mma_tf32_ss(d_tmem, smem_desc_sw128(sq_lo + off, 16, 1024), b, idesc, 1);
    } else {
      mma_bf16_ss(d_tmem, a, b, idesc, kk > 0);
    }
  }
}

// fp32 variant: row `r` of a [128, D] fp32 tile (128-byte swizzled boxes) is
// replaced by its tf32 rounding (nearest, ties away) and the remainder is
// written at the same position of `lo`.
template <int D>
__device__ __forceinline__ void split_tf32_row(uint32_t tile, uint32_t lo, int r) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 4) {
    const uint32_t off = swz128((c0 / 32) * kBoxBytes, r, (c0 % 32) / 4);
    float x[4];
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3])
                 : "r"(tile + off) : "memory");
    uint32_t hi[4];
    float rem[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi[e]) : "f"(x[e]));
      rem[e] = x[e] - __uint_as_float(hi[e]);
    }
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(tile + off), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]),
                 "r"(hi[3]) : "memory");
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" :: "r"(lo + off), "f"(rem[0]), "f"(rem[1]), "f"(rem[2]),
                 "f"(rem[3]) : "memory");
  }
}

template <typename T, int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t sv, uint32_t idesc, bool acc) {
  using C = FwdCfg<T, D>;
  // bf16: V tile is [keys, d] with d contiguous, an MN-major B operand: leading
  // byte offset = distance between 128-byte column chunks (one TMA box), stride
  // byte offset = distance between 8-key groups. tf32: sv = V^T [d rows, 128
  // keys], K-major, four boxes of 32 keys, each D rows x 128 bytes.
  const uint64_t vd = C::kTf32 ? smem_desc_sw128(sv, 16, 1024) : smem_desc_sw128(sv, kBoxBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < kBN / C::kUmmaK; ++kk) {
    const uint32_t a = p_tmem + kk * 8;                       // 8 TMEM columns per K step
    if constexpr (C::kTf32) {
      const uint32_t kb = kk * 32;
      mma_tf32_ts(d_tmem, a, desc_add(vd, (kb / 128) * (D * 128) + (kb % 128)), idesc, acc || kk > 0);
    } else {
      mma_bf16_ts(d_tmem, a, desc_add(vd, kk * C::kUmmaK * 128), idesc, acc || kk > 0);
    }
  }
}

template <typename T, int D, bool kSparse>
__global__ void __launch_bounds__(FwdCfg<T, D>::kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
           const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
           const FwdParams p) {
  using C = FwdCfg<T, D>;
  // the block-sparse variant gives one ring slot to its list of key tiles
  constexpr int kSt = kSparse ? C::kStages - 1 : C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);

  const uint32_t s_q[2] = {base, base + C::kTileBytes};
  const uint32_t s_kv = base + 2 * C::kTileBytes;
  // fp32 only: low tf32 parts of Q and of the K tile being used (after the ring)
  const uint32_t s_q_lo = s_kv + kSt * C::kTileBytes;
  const uint32_t s_k_lo = s_q_lo + C::kTileBytes;
  const uint32_t bars = s_kv + (kSt + (C::kTf32 ? 2 : 0)) * C::kTileBytes;
  auto bar_q_full = [&](int i) { return bars + 8u * i; };                       // 2
  auto bar_kv_full = [&](int s) { return bars + 16u + 8u * s; };               // kStages
  auto bar_kv_empty = [&](int s) { return bars + 16u + 8u * (kSt + s); };
  auto bar_s_full = [&](int i) { return bars + 16u + 16u * kSt + 8u * i; };
  auto bar_p_ready = [&](int i) { return bars + 32u + 16u * kSt + 8u * i; };
  auto bar_o_final = [&](int i) { return bars + 48u + 16u * kSt + 8u * i; };
  const uint32_t bar_qk_ready = bars + 64u + 16u * kSt;          // fp32: Q and K_0 split
  uint8_t* const gbars = gbase + (bars - base);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbars + 72 + 16 * kSt);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbars + 76 + 16 * kSt);
  // block-sparse: the key tiles either query tile may see, ascending, after the
  // barriers; entry = tile | (visible to tile 0) << 14 | (visible to tile 1) << 15
  int* const list_count = reinterpret_cast<int*>(gbars + 480);       // [0] all, [1] group 0's prefix
  const uint32_t bar_stall = bars + 472;                             // nothing arrives (timeout test)
  unsigned long long* const clock_start = reinterpret_cast<unsigned long long*>(gbars + 456);   // [2]
  static_assert(80 + 16 * C::kStages <= 456, "barrier area");
  uint16_t* const tile_list = reinterpret_cast<uint16_t*>(gbars + C::kBarBytes);

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
  const int qt[2] = {C::kTilesPerCta * pair, C::kTilesPerCta * pair + 1};
  // key tiles a query tile reaches: causal, up to the one holding key
  // (last row + Nk - N), none if that is negative
  auto reach = [&](int t) {
    if (!p.causal) return nk;
    const int last = t * kBM + kBM - 1 + p.causal_off;
    return last < 0 ? 0 : min(nk, last / kBN + 1);
  };
  int nkv[2];
  nkv[0] = reach(qt[0]);
  nkv[1] = (C::kPingPong && qt[1] < nq) ? reach(qt[1]) : 0;
  const bool has_tile[2] = {true, C::kPingPong && qt[1] < nq};

  if (threadIdx.x == 0) {
    clock_mark(clock_start);
    *abort_flag = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_q_full(i), 1);
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_p_ready(i), C::kPingPong ? 129 : 128);   // + the ring watcher (bf16)
      mbar_init(bar_o_final(i), 1);
    }
    for (int s = 0; s < kSt; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    mbar_init(bar_qk_ready, 128);
    mbar_init(bar_stall, 1);
    fence_mbar_init();
  }
  if constexpr (kSparse) {
    if (warp == 0) {
      // compact the key tiles visible to either query tile (within its causal
      // range) into the list, 32 candidates per round
      const unsigned char* m0 = p.mask + static_cast<long long>(b) * p.mask_sb +
                                static_cast<long long>(h) * p.mask_sh + static_cast<long long>(qt[0]) * p.mask_nt;
      const unsigned char* m1 = m0 + p.mask_nt;
      const int nscan = nkv[0] > nkv[1] ? nkv[0] : nkv[1];
      int count = 0, count0 = 0;
      for (int base0 = 0; base0 < nscan; base0 += 32) {
        const int jj = base0 + lane;
        const bool a0 = jj < nkv[0] && m0[jj] != 0;
        const bool a1 = jj < nkv[1] && m1[jj] != 0;
        const unsigned bal = __ballot_sync(0xffffffffu, a0 || a1);
        const unsigned bal0 = __ballot_sync(0xffffffffu, (a0 || a1) && jj < nkv[0]);
        if (a0 || a1)
          tile_list[count + __popc(bal & ((1u << lane) - 1u))] =
              static_cast<uint16_t>(jj | (a0 ? 1 << 14 : 0) | (a1 ? 1 << 15 : 0));
        count += __popc(bal);
        count0 += __popc(bal0);
      }
      if (lane == 0) {
        list_count[0] = count;
        list_count[1] = count0;
      }
    }
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
  if constexpr (kSparse) {
    // steps now index the list; group 0 takes the prefix inside its causal range
    nkv[0] = list_count[1];
    nkv[1] = has_tile[1] ? list_count[0] : 0;
  }
  const int nmax = nkv[0] > nkv[1] ? nkv[0] : nkv[1];
  // key tile of step j
  auto kv_tile = [&](int j) -> int { return kSparse ? (tile_list[j] & 0x3FFF) : j; };

  if (warp == C::kProd) {
    // ------------------------------------------------------------ producer
    if constexpr (C::kPingPong) setmaxnreg_dec<C::kRegsOther>();
    if (lane == 0) {
      tma_prefetch_map(&map_q);
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      for (int i = 0; i < 2; ++i) {
        if (nkv[i] == 0) continue;
        mbar_arrive_expect_tx(bar_q_full(i), C::kTileBytes);
        for (int bx = 0; bx < C::kNBox; ++bx)
          tma_load_3d(s_q[i] + bx * kBoxBytes, &map_q, bar_q_full(i), bx * C::kChunk, qt[i] * kBM, bh);
      }
      for (int c = 0; c < 2 * nmax; ++c) {
        const int slot = c % kSt;
        const uint32_t round = c / kSt;
        if (!mbar_wait(bar_kv_empty(slot), (round & 1u) ^ 1u, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_kv_full(slot), C::kTileBytes);
        const CUtensorMap* m = (c & 1) ? &map_v : &map_k;
        const uint32_t dst = s_kv + slot * C::kTileBytes;
        for (int bx = 0; bx < C::kNBox; ++bx)
          tma_load_3d(dst + bx * kBoxBytes, m, bar_kv_full(slot), bx * C::kChunk, kv_tile(c >> 1) * kBN, bh_kv);
      }
    }
    __syncwarp();
  } else if (warp == C::kIss) {
    // ------------------------------------------------------------ tensor-core issuer
    if constexpr (C::kPingPong) setmaxnreg_dec<C::kRegsOther>();
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(C::kFmt, 128, 128, 0, 0);
      const uint32_t idesc_pv = make_idesc(C::kFmt, 128, D, 0, C::kTf32 ? 0 : 1);
      const uint32_t s_vt = s_q[1];                 // V^T buffer of the fp32 variant
      bool ok = true;
      if (p.test_stall) ok = mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      for (int i = 0; i < 2 && ok; ++i)
        if (nkv[i] > 0) ok = mbar_wait(bar_q_full(i), 0, abort_flag, deadline);
      int c = 0;
      auto take = [&](uint32_t& slot_addr, int& slot) -> bool {
        slot = c % kSt;
        const bool r = mbar_wait(bar_kv_full(slot), (c / kSt) & 1, abort_flag, deadline);
        slot_addr = s_kv + slot * C::kTileBytes;
        ++c;
        return r;
      };
      uint32_t sk = 0;
      int kslot = 0;
      if (ok && nmax > 0) ok = take(sk, kslot);     // (a block-sparse CTA may have no key tile)
      if (ok && C::kTf32) ok = mbar_wait(bar_qk_ready, 0, abort_flag, deadline);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < 2; ++i) {
          if (nkv[i] == 0) continue;
          issue_qk<T, D>(tbase + C::col_s(i), s_q[i], sk, idesc_qk, s_q_lo, s_k_lo);
          mma_commit(bar_s_full(i));
        }
        if constexpr (!C::kPingPong) mma_commit(bar_kv_empty(kslot));
      }
      for (int j = 0; j < nmax && ok; ++j) {
        uint32_t sv = 0, sk_next = 0;
        int vslot = 0, knext = 0;
        const bool has_next = j + 1 < nmax;
        if constexpr (C::kPingPong) {
          // residency of V_j and K_{j+1} is folded into the P-ready barriers
          vslot = c % kSt;
          sv = s_kv + vslot * C::kTileBytes;
          ++c;
          if (has_next) {
            knext = c % kSt;
            sk_next = s_kv + knext * C::kTileBytes;
            ++c;
          }
        } else {
          ok = take(sv, vslot);
          if (ok && has_next) ok = take(sk_next, knext);
          if (!ok) break;
        }
        for (int i = 0; i < 2; ++i) {
          if (j >= nkv[i]) continue;
          if (!mbar_wait(bar_p_ready(i), j & 1, abort_flag, deadline)) { ok = false; break; }
          tc_fence_after();
          issue_pv<T, D>(tbase + C::col_o(i), tbase + C::col_s(i), C::kTf32 ? s_vt : sv, idesc_pv, j > 0);
          if (j + 1 < nkv[i]) {
            issue_qk<T, D>(tbase + C::col_s(i), s_q[i], sk_next, idesc_qk, s_q_lo, s_k_lo);
            mma_commit(bar_s_full(i));
          } else {
            mma_commit(bar_o_final(i));
          }
        }
        if (!ok) break;
        if constexpr (!C::kPingPong) {
          mma_commit(bar_kv_empty(vslot));
          if (has_next) mma_commit(bar_kv_empty(knext));
        }
      }
    }
    __syncwarp();
  } else if (C::kPingPong && warp >= 10) {
    // ------------------------------------------------------------ ring watcher (bf16; warp 11 idle)
    setmaxnreg_dec<C::kRegsOther>();
    if (warp == 10 && lane == 0) {
      // L: the group whose S MMAs are issued last in each step (group 1 unless absent)
      const int L = (nkv[1] == nmax) ? 1 : 0;
      // parity waits only tell phase k from phase k-1: observe every phase of
      // every slot in order, starting with K_0 (load 0), which only the
      // issuer needs
      bool ok = nmax == 0 || mbar_wait(bar_kv_full(0), 0, abort_flag, deadline);
      auto hand_p = [&](int i, int j) {
        // arrive for phase j only once phase j-1 has completed
        if (j > 0) ok = mbar_wait(bar_p_ready(i), (j - 1) & 1, abort_flag, deadline);
        if (ok) mbar_arrive(bar_p_ready(i));
      };
      for (int j = 0; j < nmax && ok; ++j) {
        // step j reads V_j (load 2j+1) and, if there is a next tile, K_{j+1} (load 2j+2)
        const int cv = 2 * j + 1;
        ok = mbar_wait(bar_kv_full(cv % kSt), (cv / kSt) & 1, abort_flag, deadline);
        if (ok && j + 1 < nmax) {
          const int ck = 2 * j + 2;
          ok = mbar_wait(bar_kv_full(ck % kSt), (ck / kSt) & 1, abort_flag, deadline);
        }
        if (ok && L == 1 && j < nkv[0]) hand_p(0, j);
        // S_L(j) done: it was issued after every MMA that reads K_j or V_{j-1},
        // and the tensor core completes one thread's MMAs in order. Waited for
        // before P-ready(L) phase j is handed, so this barrier cannot be two
        // phases ahead of the parity asked for.
        if (ok) ok = mbar_wait(bar_s_full(L), j & 1, abort_flag, deadline);
        if (ok) {
          mbar_arrive(bar_kv_empty((2 * j) % kSt));
          if (j > 0) mbar_arrive(bar_kv_empty((2 * j - 1) % kSt));
        }
        if (ok) hand_p(L, j);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax groups
    if constexpr (C::kPingPong) setmaxnreg_inc<C::kRegsSoftmax>();
    const int g = (warp - C::kSm0) >> 2;           // 0 or 1
    const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;           // query row within the tile
    const int n_kv = nkv[g];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tbase + lane_off + C::col_s(g);
    const uint32_t t_o = tbase + lane_off + C::col_o(g);
    const int q_row = qt[g] * kBM + row;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;                           // running max, log2 units of scale*s
    float l = 0.f;                                 // running sum relative to m
    bool ok = n_kv > 0;
    if constexpr (C::kTf32) {
      if (ok) {
        // split this thread's Q row and K_0 row (load 0 of the ring) into tf32 high + low parts
        bool w = mbar_wait(bar_q_full(0), 0, abort_flag, deadline) &&
                 mbar_wait(bar_kv_full(0), 0, abort_flag, deadline);
        ok = __all_sync(0xffffffffu, w);
        if (ok) {
          split_tf32_row<D>(s_q[0], s_q_lo, row);
          split_tf32_row<D>(s_kv, s_k_lo, row);
          fence_proxy_async_smem();
          mbar_arrive(bar_qk_ready);
        }
      }
    }
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

      // mask: causal diagonal tile and the ragged tail of the key range
      int lim = kBN;
      const int kvt = kv_tile(j);
      const int kv0 = kvt * kBN;
      if (p.causal) lim = min(lim, q_row + p.causal_off - kv0 + 1);   // bottom-right: key <= row + Nk - N
      if (kv0 + kBN > p.Nk) lim = min(lim, p.Nk - kv0);
      if (kSparse && !((tile_list[j] >> (14 + g)) & 1)) lim = 0;   // tile visible to the other query tile only
      if (lim < kBN) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      // row max: four independent chains of three-input max over 32 logits each
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
      if constexpr (C::kTf32) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t pr[32];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float p0 = ex2_approx(fmaf(s[q4 * 32 + c], sl2, neg_m));
            const float p1 = ex2_approx(fmaf(s[q4 * 32 + c + 1], sl2, neg_m));
            sum0 += p0;
            sum1 += p1;
            pr[c] = __float_as_uint(p0);
            pr[c + 1] = __float_as_uint(p1);
          }
          tmem_st_32x32b_x32(t_s + q4 * 32, pr);
        }
      } else {
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
      }
      l = l * alpha + (sum0 + sum1);
      if constexpr (C::kTf32) {
        // V_j (load 2j+1 of the ring) -> V^T in K-major 128-byte-swizzled boxes
        const int cv = 2 * j + 1;
        const int vslot = cv % kSt;
        bool vok = mbar_wait(bar_kv_full(vslot), (cv / kSt) & 1, abort_flag, deadline);
        vok = __all_sync(0xffffffffu, vok);
        if (!vok) { ok = false; break; }
        const uint32_t sv = s_kv + vslot * C::kTileBytes;
        const uint32_t svt = s_q[1];
        const int key = row;                          // this thread moves key row `key`
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 4) {
          float4 x;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                       : "r"(swz128(sv + (c0 / 32) * kBoxBytes, key, (c0 % 32) / 4)) : "memory");
          const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = c0 + e;
            const uint32_t dst = swz128(svt + (key / 32) * (D * 128), c, (key % 32) / 4) + (key % 4) * 4;
            asm volatile("st.shared.f32 [%0], %1;" :: "r"(dst), "f"(xv[e]) : "memory");
          }
        }
        if (j + 1 < n_kv) {
          // K_{j+1} (load 2j+2): split before the tensor core computes S_{j+1}. The
          // previous S, which read the low-part buffer, has completed.
          const int ck = 2 * j + 2;
          const int kslot = ck % kSt;
          bool kok = mbar_wait(bar_kv_full(kslot), (ck / kSt) & 1, abort_flag, deadline);
          kok = __all_sync(0xffffffffu, kok);
          if (!kok) { ok = false; break; }
          split_tf32_row<D>(s_kv + kslot * C::kTileBytes, s_k_lo, row);
        }
        fence_proxy_async_smem();
      }
      // O <- alpha O before the next P V accumulates. The previous P V of this
      // tile has completed: it was issued before the S MMA whose completion we
      // just waited for, and the tensor core completes them in order.
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
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
      mbar_arrive(bar_p_ready(g));
    }
    // ---------------------------------------------------------- epilogue
    // A query tile that sees no key tile at all (block mask, or more queries
    // than keys under the causal rule) skips the loop and writes O = 0,
    // LSE = -inf; so does any row that saw no key (l = 0).
    const bool empty = has_tile[g] && n_kv == 0;
    if (ok) {
      ok = mbar_wait(bar_o_final(g), 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok || empty) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.0f / l : 0.f;
      const uint32_t stage = s_q[g];     // Q tile no longer needed: all its MMAs completed
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
        if constexpr (C::kTf32) {
          const uint32_t box = stage + (c0 / 32) * kBoxBytes;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 v = make_float4(__uint_as_float(o[4 * u]) * inv_l, __uint_as_float(o[4 * u + 1]) * inv_l,
                                         __uint_as_float(o[4 * u + 2]) * inv_l, __uint_as_float(o[4 * u + 3]) * inv_l);
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, row, u)),
                         "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
          }
        } else {
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
      }
      fence_proxy_async_smem();
      if (q_row < p.N) p.lse[static_cast<size_t>(bh) * p.N + q_row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
    // every warp of the group meets here whether or not its waits succeeded,
    // so a timeout in one warp cannot leave the others stuck on the barrier;
    // a warp that gave up has raised the abort flag, and then nothing is stored
    named_bar_sync(1 + g, 128);
    if (has_tile[g] && !*abort_flag && warp == C::kSm0 + 4 * g && lane == 0) {
      for (int bx = 0; bx < C::kNBox; ++bx)
        tma_store_3d(&map_o, s_q[g] + bx * kBoxBytes, bx * C::kChunk, qt[g] * kBM, bh);
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
  if (threadIdx.x == 0) clock_record(p.clock_acc, clock_start);
}

template <typename T, int D, bool kSparse>
static cudaError_t launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                          const FwdParams& p, int grid, cudaStream_t stream) {
  using C = FwdCfg<T, D>;
  // the block-sparse variant: one ring slot fewer, the tile list after the barriers
  constexpr int kSmem = kSparse ? C::kSmemBytes - C::kTileBytes + 2 * kMaskMaxTiles : C::kSmemBytes;
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    return cudaFuncSetAttribute(fwd_kernel<T, D, kSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (e != cudaSuccess) return e;
  fwd_kernel<T, D, kSparse><<<grid, C::kThreads, kSmem, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int dtype_bytes, int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mo, FwdParams p, cudaStream_t stream) {
  const int nq = (p.N + kBM - 1) / kBM;
  p.num_pairs = (dtype_bytes == 2) ? (nq + 1) / 2 : nq;    // query tiles per CTA: 2 (bf16) or 1 (fp32)
  const int grid = p.num_pairs * p.BH;
  const bool sparse = p.mask != nullptr;
  if (sparse && (dtype_bytes != 2 || nq > kMaskMaxTiles)) return cudaErrorInvalidValue;
  // d < 128 runs in the kernel for the next size up: TMA fills the columns
  // past d with zeros on load and skips them on store
  if (dtype_bytes == 2 && d > 64 && d <= 128)
    return sparse ? launch<__nv_bfloat16, 128, true>(mq, mk, mv, mo, p, grid, stream)
                  : launch<__nv_bfloat16, 128, false>(mq, mk, mv, mo, p, grid, stream);
  if (dtype_bytes == 2 && d <= 64)
    return sparse ? launch<__nv_bfloat16, 64, true>(mq, mk, mv, mo, p, grid, stream)
                  : launch<__nv_bfloat16, 64, false>(mq, mk, mv, mo, p, grid, stream);
  if (dtype_bytes == 4 && d == 64) return launch<float, 64, false>(mq, mk, mv, mo, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
