// Backward exact attention on sm_103a: dQ, dK, dV of <O, dO> recomputed from
// the stored logsumexp.
//
// Method: the forward keeps only O and the softmax normaliser and the
// backward recomputes the probabilities from it ("4.3 FlashAttention-2与
// FlashAttention-3演进", FlashAttention-3 section 3); the backward is blockwise
// like the forward (deepschool.ru FlashAttention-2, "Улучшение backward pass");
// dQ is accumulated with asynchronous fp32 atomic adds in wide transactions
// ("Flash Attention V3技术解析" 2.1, "梯度计算").
//
// Three launches on one stream:
//  1. bwd_pre_kernel   D_i = sum_c dO_ic O_ic, LSE_i * log2(e) into a padded
//                      per-tile layout (padding: D = 0, LSE = +inf so that the
//                      padded query rows get P = 0), and dQacc = 0.
//  2. bwd_dkdv_kernel  one CTA per 128-key tile of one (batch, KV head). For
//                      each query head of the group and each query tile that
//                      can see these keys:
//                        S^T  = K Q_i^T            (TMEM)
//                        dP^T = V dO_i^T           (TMEM)
//                        P^T  = 2^(S^T s log2e - LSE_i log2e)   (registers -> TMEM, bf16)
//                        dS^T = P^T (dP^T - D_i)   (registers -> shared memory, bf16)
//                        dV  += P^T dO_i,  dK += dS^T Q_i      (TMEM accumulators)
//                        dQ_i = dS K               (TMEM -> shared -> TMA reduce-add into dQacc)
//                      and finally dK *= scale; dK, dV stored once (deterministic).
//  3. bwd_dq_kernel    dQ = scale * dQacc -> bf16.
#include <algorithm>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

// ------------------------------------------------------------------ preprocess
// One 16-lane group per row (d = 128: 8 bf16 per lane; d = 64: 4 per lane;
// D = 0: any other d, one element per lane and step).
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      const float* __restrict__ lse, BwdParams p, int d) {
  constexpr int kPer = D / 16;
  const int tid = blockIdx.x * blockDim.x + threadIdx.x;
  const int nthreads = gridDim.x * blockDim.x;
  const long long rows = static_cast<long long>(p.BH) * p.NQP;
  // each warp takes two rows per iteration (one per half-warp); the loop trip
  // count is uniform across the warp so the shuffles below see every lane
  for (long long w = tid / 32; 2 * w < rows; w += nthreads / 32) {
    const long long r = 2 * w + ((tid >> 4) & 1);
    const bool valid_row = r < rows;
    const int bh = valid_row ? static_cast<int>(r / p.NQP) : 0;
    const int i = valid_row ? static_cast<int>(r % p.NQP) : p.N;
    float acc = 0.f;
    if (i < p.N && D == 0) {
      const size_t row0 = (static_cast<size_t>(bh) * p.N + i) * d;
      for (int c = tid & 15; c < d; c += 16)
        acc = fmaf(__bfloat162float(o[row0 + c]), __bfloat162float(dO[row0 + c]), acc);
    } else if (i < p.N) {
      const size_t off = (static_cast<size_t>(bh) * p.N + i) * D + (tid & 15) * kPer;
      if constexpr (kPer == 8) {
        const uint4 a = *reinterpret_cast<const uint4*>(o + off);
        const uint4 b = *reinterpret_cast<const uint4*>(dO + off);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(a2[e]);
          const float2 y = __bfloat1622float2(b2[e]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
      } else {
        const uint2 a = *reinterpret_cast<const uint2*>(o + off);
        const uint2 b = *reinterpret_cast<const uint2*>(dO + off);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 x = __bfloat1622float2(a2[e]);
          const float2 y = __bfloat1622float2(b2[e]);
          acc = fmaf(x.x, y.x, acc);
          acc = fmaf(x.y, y.y, acc);
        }
      }
    }
#pragma unroll
    for (int s = 8; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if ((tid & 15) == 0 && valid_row) {
      p.ws_d[r] = acc;
      p.ws_lse2[r] = (i < p.N) ? lse[static_cast<size_t>(bh) * p.N + i] * kLog2e : INFINITY;
    }
  }
  // the dQ accumulator, when the workspace has one (the deterministic
  // backward's workspace holds only the LSE and D parts: ws_dq is null)
  if (p.ws_dq == nullptr) return;
  const long long n4 = static_cast<long long>(p.BH) * p.N * d / 4;
  float4* acc4 = reinterpret_cast<float4*>(p.ws_dq);
  for (long long x = tid; x < n4; x += nthreads) acc4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------ dQ convert
__global__ void __launch_bounds__(256) bwd_dq_kernel(__nv_bfloat16* __restrict__ dq, BwdParams p, int d) {
  const long long n8 = static_cast<long long>(p.BH) * p.N * d / 8;     // d is a multiple of 8
  const float4* src = reinterpret_cast<const float4*>(p.ws_dq);
  uint4* dst = reinterpret_cast<uint4*>(dq);
  const float s = p.scale;
  for (long long x = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; x < n8;
       x += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = src[2 * x], b = src[2 * x + 1];
    uint4 r;
    r.x = pack_bf16x2(a.x * s, a.y * s);
    r.y = pack_bf16x2(a.z * s, a.w * s);
    r.z = pack_bf16x2(b.x * s, b.y * s);
    r.w = pack_bf16x2(b.z * s, b.w * s);
    dst[x] = r;
  }
}

// ------------------------------------------------------------------ dK / dV
// Shared memory: K | V | dS^T | stage0 {Q, dO} | stage1 {Q, dO} | LSE[2] | D[2] | barriers.
// dQ_i (fp32, 128 rows x D) leaves through shared memory in two halves, one
// per softmax-gradient group, written over step i's own stage once its
// readers are done: columns [0, D/2) over Q_i (read by S^T_i and dK_i),
// [D/2, D) over dO_i (read by dP^T_i and dV_i). The reducer sends the Q-side
// half first, since Q_{i+2} is needed earlier in step i+2 than dO_{i+2}; the
// reductions run at the L2's fp32 reduce rate (about 23 bytes per cycle per
// SM with every SM reducing), so each half holds its region ~1600 cycles.
template <int D>
struct BwdCfg {
  static constexpr int kNBox = D / 64;                 // bf16: 64 elements per 128-byte row
  static constexpr int kTileBytes = kNBox * kBoxBytes;  // one [128, D] bf16 tile
  static constexpr int kDsBytes = 2 * kBoxBytes;       // dS^T [128 keys, 128 queries] bf16
  static constexpr int kVecBytes = 512;                // 128 fp32 (LSE or D of one query tile)
  static constexpr int kDqHalfBoxes = D / 64;          // fp32 boxes of 32 columns in D/2 columns
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffDs = 2 * kTileBytes;
  static constexpr int kOffStage = kOffDs + kDsBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffVec = kOffStage + 2 * kStageBytes;
  static constexpr int kOffBar = kOffVec + 4 * kVecBytes;
  static constexpr int kLayoutBytes = kOffBar + 256;
  static constexpr int kSmemAlloc = 232448;            // the per-block maximum; the base is aligned inside it
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
  // producer, MMA, 8 softmax-gradient warps, dQ reducer, ring watcher
  static constexpr int kThreads = 384;
  static_assert(kLayoutBytes <= kSmemAlloc, "shared memory budget");
  static_assert(2 * D + 256 <= 512, "TMEM budget");
  static_assert(kDqHalfBoxes * kBoxBytes <= kDsBytes && kDqHalfBoxes * kBoxBytes <= kTileBytes, "dQ staging");
};

template <int D, bool kSparse>
__global__ void __launch_bounds__(384, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
                const __grid_constant__ CUtensorMap map_dqacc, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  if ((base - raw) + C::kLayoutBytes > static_cast<uint32_t>(C::kSmemAlloc)) {
    // The layout needs the dynamic window to start within 768 bytes of a
    // 1 KB boundary; refuse (and report) rather than overrun.
    if (threadIdx.x == 0) atomicOr(p.status, kDevLayout);
    return;
  }
  const uint32_t s_k = base + C::kOffK, s_v = base + C::kOffV, s_ds = base + C::kOffDs;
  auto s_q = [&](int st) { return base + C::kOffStage + st * C::kStageBytes; };
  auto s_do = [&](int st) { return base + C::kOffStage + st * C::kStageBytes + C::kTileBytes; };
  auto s_lse = [&](int st) { return base + C::kOffVec + st * C::kVecBytes; };
  auto s_dvec = [&](int st) { return base + C::kOffVec + (2 + st) * C::kVecBytes; };
  const uint32_t bars = base + C::kOffBar;
  const uint32_t bar_kv_full = bars;
  auto bar_q_full = [&](int st) { return bars + 8u + 8u * st; };       // Q, LSE, D of the step
  auto bar_do_full = [&](int st) { return bars + 24u + 8u * st; };
  auto bar_q_empty = [&](int st) { return bars + 40u + 8u * st; };     // regions read out by the reducer
  auto bar_do_empty = [&](int st) { return bars + 56u + 8u * st; };
  // per softmax group, stage and 32-column fp32 box: the reducer starts on a
  // box as soon as it is written; a group cannot stage the same stage again
  // before the reducer has taken the previous use, so parities never alias
  auto bar_dq_staged = [&](int g, int st, int bx) { return bars + 72u + 8u * (4 * g + 2 * st + bx); };
  const uint32_t bar_s_full = bars + 136, bar_dp_full = bars + 144, bar_p_ready = bars + 152;
  const uint32_t bar_ds_ready = bars + 160, bar_dq_full = bars + 168, bar_dq_free = bars + 176;
  const uint32_t bar_o_final = bars + 184;
  const uint32_t bar_dk_done = bars + 216;                 // dK_i complete: Q_i may be overwritten
  const uint32_t bar_stall = bars + 208;                   // nothing arrives (timeout test)
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 192);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 196);
  unsigned long long* const clock_start = reinterpret_cast<unsigned long long*>(gbase + C::kOffBar + 224);   // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: (key tile, batch * kv head). KV heads go in groups of
  // p.head_group whose Q, dO and fp32 dQ accumulator fit in part of L2; in a
  // group the key tiles with the most query tiles to visit (small index when
  // causal) go first. `cta` is the item's logical index, key tile * BHkv +
  // batch * Hkv + kv head (the block-sparse step lists are kept by it).
  const int nkt = p.NKP / kBN;
  const int grp = blockIdx.x / (nkt * p.head_group);
  const int gsize = min(p.head_group, p.BHkv - grp * p.head_group);
  const int local = blockIdx.x - grp * p.head_group * nkt;
  const int jt = local / gsize;
  const int bhkv = grp * p.head_group + local % gsize;
  const int cta = jt * p.BHkv + bhkv;
  const int b = bhkv / p.Hkv, hk = bhkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int nq = p.NQP / kBM;
  // first query tile that sees key tile jt: causal, the one holding query
  // row jt*128 - (Nk - N) (bottom-right alignment; jt itself when Nk == N)
  const int first_row = jt * kBN - p.causal_off;
  const int it0 = p.causal ? (first_row <= 0 ? 0 : min(nq, first_row / kBM)) : 0;
  const int tiles_per_head = nq - it0;
  // block-sparse: only the (head, query tile) steps the mask lets see this key
  // tile, in the dense order, from the list bwd_blocklist_kernel compacted
  const int nsteps = kSparse ? p.ws_count[cta] : G * tiles_per_head;
  const unsigned* const steps = kSparse ? p.ws_list + static_cast<size_t>(cta) * G * nq : nullptr;

  if (threadIdx.x == 0) {
    clock_mark(clock_start);
    *abort_flag = 0;
    mbar_init(bar_kv_full, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(bar_q_full(st), 1);
      mbar_init(bar_do_full(st), 1);
      mbar_init(bar_q_empty(st), 1);
      mbar_init(bar_do_empty(st), 1);
      for (int bx = 0; bx < C::kDqHalfBoxes; ++bx) {
        mbar_init(bar_dq_staged(0, st, bx), 128);
        mbar_init(bar_dq_staged(1, st, bx), 128);
      }
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_p_ready, 256);
    mbar_init(bar_ds_ready, 256);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_free, 257);           // + the watcher: dO of the next step has landed
    mbar_init(bar_o_final, 1);
    mbar_init(bar_dk_done, 1);
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
  auto step_head = [&](int step) {
    return b * p.Hq + hk * G + (kSparse ? static_cast<int>(steps[step] >> 16) : step / tiles_per_head);
  };
  auto step_tile = [&](int step) {
    return kSparse ? static_cast<int>(steps[step] & 0xFFFFu) : it0 + step % tiles_per_head;
  };

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
        const uint32_t par = ((step >> 1) & 1) ^ 1;
        const int bh = step_head(step), it = step_tile(step);
        if (!mbar_wait(bar_q_empty(st), par, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_q_full(st), C::kTileBytes + 2 * C::kVecBytes);
        for (int bx = 0; bx < C::kNBox; ++bx)
          tma_load_3d(s_q(st) + bx * kBoxBytes, &map_q, bar_q_full(st), bx * 64, it * kBM, bh);
        const size_t voff = static_cast<size_t>(bh) * p.NQP + static_cast<size_t>(it) * kBM;
        bulk_load(s_lse(st), p.ws_lse2 + voff, C::kVecBytes, bar_q_full(st));
        bulk_load(s_dvec(st), p.ws_d + voff, C::kVecBytes, bar_q_full(st));
        if (!mbar_wait(bar_do_empty(st), par, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(bar_do_full(st), C::kTileBytes);
        for (int bx = 0; bx < C::kNBox; ++bx)
          tma_load_3d(s_do(st) + bx * kBoxBytes, &map_do, bar_do_full(st), bx * 64, it * kBM, bh);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ tensor-core issuer
    // Step i: [P^T_i ready] dV, [dS^T_i ready] dQ_i then dK_i, then for step
    // i+1: [Q_{i+1} landed] S^T, [dQ_i read out of TMEM, dO_{i+1} landed] dP^T.
    // dQ_i goes first so that its read-out (on the softmax-gradient warps'
    // critical path) overlaps dK_i; the group that stages over Q_i waits for
    // dK_i, its last reader. dQ goes into the dP^T columns; one thread's MMAs
    // run in issue order, which keeps every TMEM reuse below safe.
    if (lane == 0) {
      const uint32_t id_kk = make_idesc(1, 128, 128, 0, 0);  // S^T, dP^T: both operands K-major
      const uint32_t id_kmn = make_idesc(1, 128, D, 0, 1);   // dV, dK: A K-major (or TMEM), B MN-major
      const uint32_t id_mnmn = make_idesc(1, 128, D, 1, 1);  // dQ: A = dS (MN-major view of dS^T), B = K MN-major
      // descriptors built once; each MMA only adds a compile-time offset
      const uint64_t k_kmaj = smem_desc_sw128(s_k, 16, 1024), k_mn = smem_desc_sw128(s_k, kBoxBytes, 1024);
      const uint64_t v_kmaj = smem_desc_sw128(s_v, 16, 1024);
      const uint64_t ds_kmaj = smem_desc_sw128(s_ds, 16, 1024), ds_mn = smem_desc_sw128(s_ds, kBoxBytes, 1024);
      const uint64_t q_kmaj[2] = {smem_desc_sw128(s_q(0), 16, 1024), smem_desc_sw128(s_q(1), 16, 1024)};
      const uint64_t q_mn[2] = {smem_desc_sw128(s_q(0), kBoxBytes, 1024), smem_desc_sw128(s_q(1), kBoxBytes, 1024)};
      const uint64_t do_kmaj[2] = {smem_desc_sw128(s_do(0), 16, 1024), smem_desc_sw128(s_do(1), 16, 1024)};
      const uint64_t do_mn[2] = {smem_desc_sw128(s_do(0), kBoxBytes, 1024), smem_desc_sw128(s_do(1), kBoxBytes, 1024)};
      auto issue_s = [&](int st) {                          // S^T = K Q^T
        const uint64_t qk = st ? q_kmaj[1] : q_kmaj[0];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColS, desc_add(k_kmaj, off), desc_add(qk, off), id_kk, kk > 0);
        }
        mma_commit(bar_s_full);
      };
      auto issue_dp = [&](int st) {                         // dP^T = V dO^T
        const uint64_t dok = st ? do_kmaj[1] : do_kmaj[0];
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColDP, desc_add(v_kmaj, off), desc_add(dok, off), id_kk, kk > 0);
        }
        mma_commit(bar_dp_full);
      };
      // (a block-sparse key tile may have no step at all: dK = dV = 0)
      bool ok = !p.test_stall || mbar_wait(bar_stall, 0, abort_flag, deadline);   // runs out by design
      ok = ok && (nsteps == 0 ||
                  (mbar_wait(bar_kv_full, 0, abort_flag, deadline) && mbar_wait(bar_q_full(0), 0, abort_flag, deadline)));
      if (ok && nsteps > 0) {
        tc_fence_after();
        issue_s(0);
        ok = mbar_wait(bar_do_full(0), 0, abort_flag, deadline);
        if (ok) issue_dp(0);
      }
      for (int step = 0; step < nsteps && ok; ++step) {
        const int st = step & 1;
        const uint64_t qm = st ? q_mn[1] : q_mn[0], dom = st ? do_mn[1] : do_mn[0];
        if (!mbar_wait(bar_p_ready, step & 1, abort_flag, deadline)) { ok = false; break; }
        tc_fence_after();
        // dV += P^T dO  (K = 128 queries; P^T of query q sits in S column 64*(q/64) + (q%64)/2)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a = tbase + C::kColS + 64 * (kk >> 2) + (kk & 3) * 8;
          mma_bf16_ts(tbase + C::kColDV, a, desc_add(dom, kk * 16 * 128), id_kmn, step > 0 || kk > 0);
        }
        if (!mbar_wait(bar_ds_ready, step & 1, abort_flag, deadline)) { ok = false; break; }
        tc_fence_after();
        // dQ_i = dS K  (M = queries: dS^T read MN-major; K = 128 keys), into the dP^T columns
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ss(tbase + C::kColDP, desc_add(ds_mn, kk * 16 * 128), desc_add(k_mn, kk * 16 * 128), id_mnmn, kk > 0);
        mma_commit(bar_dq_full);
        // dK += dS^T Q  (A = dS^T K-major over queries)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk * 32 / 128) * kBoxBytes + (kk * 32) % 128;
          mma_bf16_ss(tbase + C::kColDK, desc_add(ds_kmaj, off), desc_add(qm, kk * 16 * 128), id_kmn,
                      step > 0 || kk > 0);
        }
        mma_commit(bar_dk_done);
        if (step + 1 < nsteps) {
          const int sn = (step + 1) & 1;
          if (!mbar_wait(bar_q_full(sn), ((step + 1) >> 1) & 1, abort_flag, deadline)) { ok = false; break; }
          tc_fence_after();
          issue_s(sn);                                      // P^T_i in the S columns was read by dV_i
          if (!mbar_wait(bar_dq_free, step & 1, abort_flag, deadline)) { ok = false; break; }
          tc_fence_after();
          issue_dp(sn);
        }
      }
      if (ok) mma_commit(bar_o_final);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------ dQ reducer
    // Adds each staged fp32 dQ half into the global accumulator with TMA bulk
    // reductions, both halves in flight together; each region goes back to
    // the producer as soon as its half has been read.
    if (lane == 0) {
      for (int step = 0; step < nsteps; ++step) {
        const int st = step & 1;
        const int bh = step_head(step), it = step_tile(step);
        bool ok = true;
        // group 0's boxes first (its region, Q, is needed first again), each
        // box as soon as it has been written
        for (int g = 0; g < 2 && ok; ++g) {
          const uint32_t src = g ? s_do(st) : s_q(st);
          for (int bx = 0; bx < C::kDqHalfBoxes && ok; ++bx) {
            ok = mbar_wait(bar_dq_staged(g, st, bx), (step >> 1) & 1, abort_flag, deadline);
            if (!ok) break;
            tma_reduce_add_3d(&map_dqacc, src + bx * kBoxBytes, g * (D / 2) + bx * 32, it * kBM, bh);
            tma_store_commit();
          }
        }
        if (!ok) break;
        tma_store_wait_read<C::kDqHalfBoxes>();
        mbar_arrive(bar_q_empty(st));
        tma_store_wait_read0();
        mbar_arrive(bar_do_empty(st));
      }
      tma_store_wait_all0();
    }
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------------ ring watcher
    // Adds one arrival to the "dQ_i read out" barrier once dO_{i+1} has
    // landed, so the issuer learns both from a single poll before dP^T_{i+1}.
    // Parity waits only tell phase k from phase k-1, so every phase of each
    // stage's barrier is observed in order, dO_0 (which only the issuer
    // needs) included: without it, dO_2 could pass for landed while dO_0 was
    // still in flight.
    if (lane == 0) {
      bool ok = nsteps == 0 || mbar_wait(bar_do_full(0), 0, abort_flag, deadline);
      for (int step = 0; step + 1 < nsteps && ok; ++step) {
        const int sn = (step + 1) & 1;
        ok = mbar_wait(bar_do_full(sn), ((step + 1) >> 1) & 1, abort_flag, deadline);
        // arrive for phase `step` only once phase step-1 has completed
        if (ok && step > 0) ok = mbar_wait(bar_dq_free, (step - 1) & 1, abort_flag, deadline);
        if (ok) mbar_arrive(bar_dq_free);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax-gradient groups
    const int g = (warp - 2) >> 2;                 // query-column half: [64g, 64g + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // key row (TMEM lane); query row for the dQ drain
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool key_pad = jt * kBN + r >= p.Nk;     // key rows past Nk contribute nothing
    bool ok = true;
    for (int step = 0; step < nsteps && ok; ++step) {
      const int st = step & 1;
      const int it = step_tile(step);
      // causal: query q of tile `it` sees key r of tile jt iff q + lim_off >= r
      const int lim_off = it * kBM + p.causal_off - jt * kBN;
      const bool diag = p.causal && lim_off < kBN - 1;
      ok = mbar_wait(bar_q_full(st), (step >> 1) & 1, abort_flag, deadline) &&
           mbar_wait(bar_s_full, step & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(gbase + (s_lse(st) - base));
      const float* dvec = reinterpret_cast<const float*>(gbase + (s_dvec(st) - base));
      // ---- phase A: P^T = 2^(S^T s log2e - LSE log2e), written over S^T as bf16 pairs
      uint32_t sv[2][32];
      tmem_ld_32x32b_x32(tbase + lane_off + C::kColS + 64 * g, sv[0]);
      tmem_ld_32x32b_x32(tbase + lane_off + C::kColS + 64 * g + 32, sv[1]);
      tmem_wait_ld();
      reg_fence_x32(sv[0]);
      reg_fence_x32(sv[1]);
      float pf[64];
      const float4* l4 = reinterpret_cast<const float4*>(lse2 + 64 * g);
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 lv = l4[c / 4];
        fms2_b(pf[c], pf[c + 1], __uint_as_float(sv[c >> 5][c & 31]), __uint_as_float(sv[c >> 5][(c & 31) + 1]),
               sl2, lv.x, lv.y);
        fms2_b(pf[c + 2], pf[c + 3], __uint_as_float(sv[c >> 5][(c & 31) + 2]),
               __uint_as_float(sv[c >> 5][(c & 31) + 3]), sl2, lv.z, lv.w);
      }
#pragma unroll
      for (int c = 0; c < 64; ++c) pf[c] = ex2_approx(pf[c]);
      if (key_pad || diag) {
        // causal tile the diagonal crosses: query q sees key r only if q + lim_off >= r
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (key_pad || 64 * g + c + lim_off < r) pf[c] = 0.f;
      }
      uint32_t pp[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) pp[c] = pack_bf16x2(pf[2 * c], pf[2 * c + 1]);
      // P^T (bf16 pairs) into TMEM over the S^T columns this group already read
      tmem_st_32x32b_x32(tbase + lane_off + C::kColS + 64 * g, pp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p_ready);
      // ---- phase B: dS^T = P^T (dP^T - D) into shared memory (bf16); the
      // previous dS^T was last read by dK and dQ of the previous step, whose
      // completion this group waited for before draining dQ
      ok = mbar_wait(bar_dp_full, step & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[2][32];
      tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + 64 * g, dp[0]);
      tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + 64 * g + 32, dp[1]);
      tmem_wait_ld();
      reg_fence_x32(dp[0]);
      reg_fence_x32(dp[1]);
      const float4* d4 = reinterpret_cast<const float4*>(dvec + 64 * g);
      uint32_t dd[32];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 dv4 = d4[c / 4];
        float ds[4];
        dsub_mul2(ds[0], ds[1], __uint_as_float(dp[c >> 5][c & 31]), __uint_as_float(dp[c >> 5][(c & 31) + 1]),
                  dv4.x, dv4.y, pf[c], pf[c + 1]);
        dsub_mul2(ds[2], ds[3], __uint_as_float(dp[c >> 5][(c & 31) + 2]), __uint_as_float(dp[c >> 5][(c & 31) + 3]),
                  dv4.z, dv4.w, pf[c + 2], pf[c + 3]);
        dd[c / 2] = pack_bf16x2(ds[0], ds[1]);
        dd[c / 2 + 1] = pack_bf16x2(ds[2], ds[3]);
      }
      // dS^T row r, query columns [64g, 64g + 64): the eight 16-byte units of box g
      const uint32_t box = s_ds + g * kBoxBytes;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(box, r, u)),
                     "r"(dd[4 * u]), "r"(dd[4 * u + 1]), "r"(dd[4 * u + 2]), "r"(dd[4 * u + 3]) : "memory");
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_ds_ready);

      // ---- dQ_i: TMEM (lane = query row r of tile `it`, this group's D/2
      // columns) -> registers -> shared memory over Q_i (group 0) or dO_i
      // (group 1), whose MMA readers have all completed -> TMA reduce-add
      ok = mbar_wait(bar_dq_full, step & 1, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t dq[D / 2];
      if constexpr (D / 2 == 64) {
        uint32_t t2[2][32];
        tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + g * (D / 2), t2[0]);
        tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + g * (D / 2) + 32, t2[1]);
        tmem_wait_ld();
        reg_fence_x32(t2[0]);
        reg_fence_x32(t2[1]);
#pragma unroll
        for (int c = 0; c < 64; ++c) dq[c] = t2[c >> 5][c & 31];
      } else {
        uint32_t t1[32];
        tmem_ld_32x32b_x32(tbase + lane_off + C::kColDP + g * (D / 2), t1);
        tmem_wait_ld();
        reg_fence_x32(t1);
#pragma unroll
        for (int c = 0; c < 32; ++c) dq[c] = t1[c];
      }
      tc_fence_before();
      mbar_arrive(bar_dq_free);
      // group 0 stages over Q_i, which dK_i (issued after dQ_i) still reads;
      // group 1's region, dO_i, was last read by dV_i and dP^T_i, both done
      if (g == 0) {
        ok = mbar_wait(bar_dk_done, step & 1, abort_flag, deadline);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      // fp32 boxes of 32 columns x 128 rows, 128-byte swizzle, each released
      // to the reducer as soon as this group has written it
      const uint32_t dst0 = g ? s_do(st) : s_q(st);
#pragma unroll
      for (int bx = 0; bx < C::kDqHalfBoxes; ++bx) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t dst = swz128(dst0 + bx * kBoxBytes, r, u);
          const int c = 32 * bx + 4 * u;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(dst), "r"(dq[c]), "r"(dq[c + 1]),
                       "r"(dq[c + 2]), "r"(dq[c + 3]) : "memory");
        }
        fence_proxy_async_smem();
        mbar_arrive(bar_dq_staged(g, st, bx));
      }
    }
    // ---------------------------------------------------------- dK, dV epilogue
    if (ok) {
      ok = mbar_wait(bar_o_final, 0, abort_flag, deadline);
      // with no step nothing waited for K and V, whose buffers stage dK and dV
      // below: let their loads land first
      if (nsteps == 0) ok = ok && mbar_wait(bar_kv_full, 0, abort_flag, deadline);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      // staging: the V buffer for dV and the K buffer for dK (every MMA has completed)
      const uint32_t stg_v = s_v, stg_k = s_k;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float mul = which ? p.scale : 1.0f;
        const uint32_t col = which ? C::kColDK : C::kColDV;
        const uint32_t stg = which ? stg_k : stg_v;
#pragma unroll
        for (int c0 = g * (D / 2); c0 < (g + 1) * (D / 2); c0 += 32) {
          uint32_t t[32];
          if (nsteps > 0) {
            tmem_ld_32x32b_x32(tbase + lane_off + col + c0, t);
            tmem_wait_ld();
            reg_fence_x32(t);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) t[c] = 0u;
          }
          const uint32_t bx = stg + (c0 / 64) * kBoxBytes;
          const int u0 = (c0 % 64) / 8;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16x2(__uint_as_float(t[8 * u + 2 * e]) * mul, __uint_as_float(t[8 * u + 2 * e + 1]) * mul);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" :: "r"(swz128(bx, r, u0 + u)),
                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
          }
        }
      }
      fence_proxy_async_smem();
    }
    // all eight softmax-gradient warps meet here whether or not their waits
    // succeeded; a warp that gave up has raised the abort flag: store nothing
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
  if (threadIdx.x == 0) clock_record(p.clock_acc, clock_start);
}

// ------------------------------------------------------------------ launch
template <int D, bool kSparse>
static cudaError_t launch_dkdv_d(const BwdMaps& m, const BwdParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  static PerDeviceOnce attr;
  const cudaError_t e = attr.run([] {
    return cudaFuncSetAttribute(bwd_dkdv_kernel<D, kSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemAlloc);
  });
  if (e != cudaSuccess) return e;
  const int grid = (p.NKP / kBN) * p.BHkv;
  // KV heads per group: the group's Q and dO (bf16) and fp32 dQ accumulator,
  // G query heads of N x d each, within 64 MB, half of L2
  BwdParams q = p;
  const long long per_kv_head = 8LL * (p.Hq / p.Hkv) * p.N * D;
  q.head_group = static_cast<int>(std::max(1LL, std::min<long long>(p.BHkv, (64LL << 20) / per_kv_head)));
  bwd_dkdv_kernel<D, kSparse><<<grid, C::kThreads, C::kSmemAlloc, stream>>>(m.q, m.k, m.v, m.dO, m.dk, m.dv,
                                                                             m.dqacc, q);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ block list
// One warp per dK/dV CTA (key tile jt, batch b, KV head hk): compacts the
// (head in group, query tile) steps whose mask byte lets the query tile see
// key tile jt, in the order the dense kernel visits them.
__global__ void __launch_bounds__(256) bwd_blocklist_kernel(BwdParams p) {
  const int cta = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int nqt = p.NQP / kBM;
  if (cta >= nqt * p.BHkv) return;
  const int jt = cta / p.BHkv, bhkv = cta % p.BHkv;
  const int b = bhkv / p.Hkv, hk = bhkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int it0 = p.causal ? jt : 0;
  const int per_head = nqt - it0;
  const int total = G * per_head;
  unsigned* const list = p.ws_list + static_cast<size_t>(cta) * G * nqt;
  int count = 0;
  for (int base = 0; base < total; base += 32) {
    const int s = base + lane;
    bool a = false;
    unsigned e = 0;
    if (s < total) {
      const int hl = s / per_head, it = it0 + s % per_head;
      const long long off = static_cast<long long>(b) * p.mask_sb + static_cast<long long>(hk * G + hl) * p.mask_sh +
                            static_cast<long long>(it) * p.mask_nt + jt;
      a = p.mask[off] != 0;
      e = static_cast<unsigned>(it) | (static_cast<unsigned>(hl) << 16);
    }
    const unsigned bal = __ballot_sync(0xffffffffu, a);
    if (a) list[count + __popc(bal & ((1u << lane) - 1u))] = e;
    count += __popc(bal);
  }
  if (lane == 0) p.ws_count[cta] = count;
}

cudaError_t launch_bwd_blocklist(const BwdParams& p, cudaStream_t stream) {
  const long long warps = static_cast<long long>(p.NQP / kBM) * p.BHkv;
  const int blocks = static_cast<int>((warps + 7) / 8);
  bwd_blocklist_kernel<<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// The two streaming kernels (grid-stride loops, 256 threads per CTA): eight
// CTAs per SM fill its 2048 thread slots, which keeps enough 16-byte loads in
// flight to cover the memory latency (four per SM left them latency-bound).
constexpr int kStreamCtasPerSm = 8;

cudaError_t launch_bwd_pre(int d, const void* o, const void* dO, const float* lse, const BwdParams& p, int num_sms,
                           cudaStream_t stream) {
  const auto* o16 = static_cast<const __nv_bfloat16*>(o);
  const auto* do16 = static_cast<const __nv_bfloat16*>(dO);
  const int grid = num_sms * kStreamCtasPerSm;
  if (d == 128) bwd_pre_kernel<128><<<grid, 256, 0, stream>>>(o16, do16, lse, p, d);
  else if (d == 64) bwd_pre_kernel<64><<<grid, 256, 0, stream>>>(o16, do16, lse, p, d);
  else if (d >= 8 && d <= 256 && d % 8 == 0) bwd_pre_kernel<0><<<grid, 256, 0, stream>>>(o16, do16, lse, p, d);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int d, const BwdMaps& m, const BwdParams& p, cudaStream_t stream) {
  const bool sparse = p.mask != nullptr;
  // d < 128 runs in the kernel for the next size up (zero-filled columns)
  if (d > 64 && d <= 128) return sparse ? launch_dkdv_d<128, true>(m, p, stream) : launch_dkdv_d<128, false>(m, p, stream);
  if (d >= 8 && d <= 64) return sparse ? launch_dkdv_d<64, true>(m, p, stream) : launch_dkdv_d<64, false>(m, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dq(int d, void* dq, const BwdParams& p, int num_sms, cudaStream_t stream) {
  auto* dq16 = static_cast<__nv_bfloat16*>(dq);
  if (d >= 8 && d <= 128 && d % 8 == 0) bwd_dq_kernel<<<num_sms * kStreamCtasPerSm, 256, 0, stream>>>(dq16, p, d);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fa
