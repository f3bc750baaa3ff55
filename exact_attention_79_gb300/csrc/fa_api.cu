// C ABI of the attention library: argument validation, TMA tensor maps,
// kernel dispatch and the device status word. See include/fa.h.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_kernels.h"

namespace {

// Status words set by kernels whose bounded waits ran out, one per stream:
// a call launched on a stream reports to that stream's word, which
// fa_device_status(stream) reads and clears. Slot 0 is shared by the streams
// beyond the first kStatusSlots - 1 that a device sees.
constexpr int kStatusSlots = 256;
__device__ unsigned g_status_words[kStatusSlots];
// SM cycles and nanoseconds summed over the CTAs of the forward and dK/dV
// kernels since the last fa_sm_clock_mhz (diagnostic, device-wide).
__device__ unsigned long long g_clock_acc[2];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
struct DeviceState {
  std::once_flag once;
  bool arch_ok = false;
  int num_sms = 0;
  unsigned* status = nullptr;           // device address of g_status_words on this device
  unsigned long long* clock_acc = nullptr;  // device address of g_clock_acc on this device
  std::mutex mu;                        // guards the stream -> slot table below
  const void* owner[kStatusSlots] = {}; // owner[i]: the stream whose calls report to slot i (i >= 1)
  int used = 1;
};
DeviceState g_dev[kMaxDevices];

// The status word of `stream` on this device: the slot the stream was given
// the first time it was seen, or the shared slot 0 once the table is full.
unsigned* stream_slot(DeviceState& s, const void* stream) {
  std::lock_guard<std::mutex> lock(s.mu);
  for (int i = 1; i < s.used; ++i)
    if (s.owner[i] == stream) return s.status + i;
  if (s.used < kStatusSlots) {
    s.owner[s.used] = stream;
    return s.status + s.used++;
  }
  return s.status;
}

// Checks the current device once (compute capability 10.3), resolves the
// device address of the status words on it and returns the word of `stream`.
fa_status device_state(const void* stream, unsigned** status_out, int* num_sms = nullptr,
                       unsigned long long** clock_acc = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  DeviceState& s = g_dev[dev];
  std::call_once(s.once, [&s, dev] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return;
    s.arch_ok = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) s.num_sms = 0;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_words) == cudaSuccess) s.status = static_cast<unsigned*>(p);
    void* c = nullptr;
    if (cudaGetSymbolAddress(&c, g_clock_acc) == cudaSuccess) s.clock_acc = static_cast<unsigned long long*>(c);
  });
  if (!s.arch_ok) return FA_ERR_ARCH;
  if (!s.status || !s.clock_acc || s.num_sms <= 0) return FA_ERR_CUDA;
  *status_out = stream_slot(s, stream);
  if (num_sms) *num_sms = s.num_sms;
  if (clock_acc) *clock_acc = s.clock_acc;
  return FA_OK;
}

unsigned long long wait_limit_ns() {
  static unsigned long long ns = [] {
    const char* e = std::getenv("FA_WAIT_LIMIT_MS");
    long ms = e ? std::strtol(e, nullptr, 10) : 0;
    if (ms <= 0) ms = 2000;
    return static_cast<unsigned long long>(ms) * 1000000ull;
  }();
  return ns;
}

// FA_TEST_STALL=1 (read at every call): the tensor-core issuer first waits on
// a barrier nothing ever arrives on, so the bounded wait runs out and the
// call reports FA_ERR_TIMEOUT; for exercising failure detection without any
// fault. Off unless set.
int test_stall() {
  const char* e = std::getenv("FA_TEST_STALL");
  return (e && e[0] == '1') ? 1 : 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// FP8 head dimensions: multiples of 16 up to 256 (a row of one-byte codes
// must be a multiple of 16 bytes for TMA). The attention kernels are built
// for 128 and 256; a smaller d runs in the next one up, its columns past d
// read as zeros and never stored.
bool fp8_dim(int d) { return d >= 16 && d <= 256 && d % 16 == 0; }

// 3-D map over a dense [BH, N, d] tensor: dims (d, N, BH), one box = 128 rows
// by 128 bytes with 128-byte swizzle. Rows past N read as zero and are not
// written by stores.
bool make_map(CUtensorMap* m, const void* ptr, int elt_bytes, int d, int N, long long BH, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elt_bytes,
                                 static_cast<cuuint64_t>(d) * N * elt_bytes};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elt_bytes), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = elt_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elt_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUresult r = enc(m, dt, 3,
                         const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

fa_status check_sizes(int B, int Hq, int Hkv, int N, int d, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  // head dims up to 256 in steps of 8 (16-byte rows for TMA); the kernels are
  // built for 64, 128, 192 and 256 and a smaller d runs in the next one up,
  // the columns past d read as zeros and never written. The backward stops
  // at 128 (bwd_dim).
  if (d < 8 || d > 256 || d % 8 != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * Hq;
  const long long nq = (N + 127) / 128;
  if (BH > (1LL << 24) || ((nq + 1) / 2) * BH >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// The one-pass backward kernels hold dK, dV, S^T and dP^T of a 128-key tile
// in TMEM (4 x d columns of 512): up to d = 128. Above that the three-pass
// backward (fa_bwd_wide.cu) serves fa_bwd, fa_bwd_kv, fa_bwd_deterministic
// and fa_bwd_noalloc; the single phases and the block-sparse backward stop at 128.
fa_status bwd_dim(int d, bool wide_ok = false) { return d > 128 && !wide_ok ? FA_ERR_UNSUPPORTED : FA_OK; }

fa_status fwd_common(int elt, const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                     int Hkv, int N, int d, int causal, float scale, void* stream,
                     const unsigned char* mask = nullptr, long long mask_sb = 0, long long mask_sh = 0,
                     int Nk = -1, bool use_pair = false) {
  if (Nk < 0) Nk = N;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, Hq, Hkv, N, d, scale);
  if (st != FA_OK) return st;
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  if (elt == 4 && d != 64) return FA_ERR_UNSUPPORTED;
  const bool wide = d > 128;                // one query tile per CTA, V in 64-key halves
  if (wide && mask) return FA_ERR_UNSUPPORTED;
  // fa_fwd_pair: CTA pairs (cta_group::2), K loaded in 64-row halves; bf16,
  // 64 < d <= 128, dense only
  const bool pair = use_pair;
  if (pair && (elt != 2 || mask || d <= 64 || d > 128)) return FA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  unsigned long long* clock_acc = nullptr;
  st = device_state(stream, &status, nullptr, &clock_acc);
  if (st != FA_OK) return st;
  CUtensorMap mq, mk, mv, mo;
  const long long BHq = static_cast<long long>(B) * Hq, BHkv = static_cast<long long>(B) * Hkv;
  if (!make_map(&mq, q, elt, d, N, BHq) || !make_map(&mk, k, elt, d, Nk, BHkv, pair ? 64 : 128) ||
      !make_map(&mv, v, elt, d, Nk, BHkv, wide ? 64 : 128) || !make_map(&mo, o, elt, d, N, BHq))
    return FA_ERR_CUDA;
  fa::FwdParams p{};
  p.lse = lse;
  p.status = status;
  p.clock_acc = clock_acc;
  p.N = N;
  p.Nk = Nk;
  p.causal_off = Nk - N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.BH = static_cast<int>(BHq);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_limit_ns();
  p.test_stall = test_stall();
  p.mask = mask;
  p.mask_sb = mask_sb;
  p.mask_sh = mask_sh;
  p.mask_nt = (N + 127) / 128;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = wide ? fa::launch_fwd_wide(d, mq, mk, mv, mo, p, s)
                        : pair ? fa::launch_fwd_pair(mq, mk, mv, mo, p, s)
                               : fa::launch_fwd(elt, d, mq, mk, mv, mo, p, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct BwdWorkspace {
  size_t off_lse2, off_d, off_dq, total;   // off_dq: the bytes the deterministic backward needs
  size_t off_count, off_list, total_sparse;  // block-sparse: per dK/dV CTA, its step count and step list
};

BwdWorkspace bwd_workspace(int B, int Hq, int Hkv, int N, int d) {
  const size_t BH = static_cast<size_t>(B) * Hq;
  const size_t NQP = static_cast<size_t>((N + 127) / 128) * 128;
  BwdWorkspace w;
  w.off_lse2 = 0;
  w.off_d = align256(BH * NQP * 4);
  w.off_dq = w.off_d + align256(BH * NQP * 4);
  w.total = w.off_dq + align256(BH * static_cast<size_t>(N) * d * 4);
  const size_t ctas = (NQP / 128) * static_cast<size_t>(B) * Hkv;
  const size_t G = static_cast<size_t>(Hq / (Hkv > 0 ? Hkv : 1));
  w.off_count = w.total;
  w.off_list = w.off_count + align256(ctas * 4);
  w.total_sparse = w.off_list + align256(ctas * G * (NQP / 128) * 4);
  return w;
}

// Validates sizes and workspace, resolves the device, fills BwdParams. With
// lse_d_only the workspace only has to hold the LSE and D parts.
fa_status bwd_setup(int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* workspace,
                    size_t workspace_bytes, fa::BwdParams* p, int* num_sms, void* stream, bool lse_d_only = false,
                    const unsigned char* mask = nullptr, long long mask_sb = 0, long long mask_sh = 0,
                    int Nk = -1) {
  if (Nk < 0) Nk = N;
  fa_status st = check_sizes(B, Hq, Hkv, N, d, scale);
  if (st != FA_OK) return st;
  if (Nk < 1 || check_sizes(B, Hq, Hkv, Nk, d, scale) != FA_OK) return FA_ERR_INVALID_ARG;
  // above d = 128 only the three-pass backward, which needs the LSE and D parts alone
  st = bwd_dim(d, lse_d_only && !mask);
  if (st != FA_OK) return st;
  const BwdWorkspace w = bwd_workspace(B, Hq, Hkv, N, d);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < (mask ? w.total_sparse : (lse_d_only ? w.off_dq : w.total)))
    return FA_ERR_WORKSPACE;
  unsigned* status = nullptr;
  unsigned long long* clock_acc = nullptr;
  st = device_state(stream, &status, num_sms, &clock_acc);
  if (st != FA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p->ws_lse2 = reinterpret_cast<float*>(ws + w.off_lse2);
  p->ws_d = reinterpret_cast<float*>(ws + w.off_d);
  // a workspace sized for the LSE and D parts alone has no dQ accumulator:
  // nothing may write past its end
  p->ws_dq = lse_d_only ? nullptr : reinterpret_cast<float*>(ws + w.off_dq);
  p->status = status;
  p->clock_acc = clock_acc;
  p->N = N;
  p->NQP = ((N + 127) / 128) * 128;
  p->Nk = Nk;
  p->NKP = ((Nk + 127) / 128) * 128;
  p->causal_off = Nk - N;
  p->Hq = Hq;
  p->Hkv = Hkv;
  p->BH = B * Hq;
  p->BHkv = B * Hkv;
  p->causal = causal ? 1 : 0;
  p->scale = scale;
  p->scale_log2 = scale * 1.4426950408889634f;
  p->timeout_ns = wait_limit_ns();
  p->test_stall = test_stall();
  p->mask = mask;
  p->mask_sb = mask_sb;
  p->mask_sh = mask_sh;
  p->mask_nt = (N + 127) / 128;
  p->ws_count = mask ? reinterpret_cast<int*>(ws + w.off_count) : nullptr;
  p->ws_list = mask ? reinterpret_cast<unsigned*>(ws + w.off_list) : nullptr;
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  if (check_sizes(B, Hq, Hkv, N, d, 1.0f) != FA_OK) return 0;
  const BwdWorkspace w = bwd_workspace(B, Hq, Hkv, N, d);
  return d > 128 ? w.off_dq : w.total;      // the three-pass backward keeps no dQ accumulator
}

size_t fa_bwd_blocksparse_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  if (check_sizes(B, Hq, Hkv, N, d, 1.0f) != FA_OK || bwd_dim(d) != FA_OK || (N + 127) / 128 > fa::kMaskMaxTiles)
    return 0;
  return bwd_workspace(B, Hq, Hkv, N, d).total_sparse;
}

fa_status fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                             const unsigned char* block_mask, long long mask_stride_b, long long mask_stride_h,
                             int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream) {
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  if (!block_mask || mask_stride_b < 0 || mask_stride_h < 0) return FA_ERR_INVALID_ARG;
  if ((N + 127) / 128 > fa::kMaskMaxTiles) return FA_ERR_UNSUPPORTED;
  fa::BwdParams p{};
  int num_sms = 0;
  fa_status st = bwd_setup(B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes, &p, &num_sms, stream, false,
                           block_mask, mask_stride_b, mask_stride_h);
  if (st != FA_OK) return st;
  fa::BwdMaps m;
  const long long BHq = static_cast<long long>(B) * Hq, BHkv = static_cast<long long>(B) * Hkv;
  if (!make_map(&m.q, q, 2, d, N, BHq) || !make_map(&m.k, k, 2, d, N, BHkv) || !make_map(&m.v, v, 2, d, N, BHkv) ||
      !make_map(&m.dO, dO, 2, d, N, BHq) || !make_map(&m.dk, dk, 2, d, N, BHkv) || !make_map(&m.dv, dv, 2, d, N, BHkv) ||
      !make_map(&m.dqacc, p.ws_dq, 4, d, N, BHq))
    return FA_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_bwd_pre(d, o, dO, lse, p, num_sms, s);
  if (e == cudaSuccess) e = fa::launch_bwd_blocklist(p, s);
  if (e == cudaSuccess) e = fa::launch_bwd_dkdv(d, m, p, s);
  if (e == cudaSuccess) e = fa::launch_bwd_dq(d, dq, p, num_sms, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd_preprocess(const void* o, const float* lse, const void* dO, void* workspace,
                            size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, void* stream) {
  if (!o || !lse || !dO || !aligned16(o) || !aligned16(lse) || !aligned16(dO)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p{};
  int num_sms = 0;
  fa_status st = bwd_setup(B, Hq, Hkv, N, d, 0, 1.0f, workspace, workspace_bytes, &p, &num_sms, stream);
  if (st != FA_OK) return st;
  const cudaError_t e = fa::launch_bwd_pre(d, o, dO, lse, p, num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

namespace {
fa_status bwd_dkdv_common(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv,
                          void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int Nk, int d,
                          int causal, float scale, void* stream) {
  const void* ptrs[] = {q, k, v, dO, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p{};
  int num_sms = 0;
  fa_status st = bwd_setup(B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes, &p, &num_sms, stream, false,
                           nullptr, 0, 0, Nk);
  if (st != FA_OK) return st;
  fa::BwdMaps m;
  const long long BHq = static_cast<long long>(B) * Hq, BHkv = static_cast<long long>(B) * Hkv;
  if (!make_map(&m.q, q, 2, d, N, BHq) || !make_map(&m.k, k, 2, d, Nk, BHkv) ||
      !make_map(&m.v, v, 2, d, Nk, BHkv) || !make_map(&m.dO, dO, 2, d, N, BHq) ||
      !make_map(&m.dk, dk, 2, d, Nk, BHkv) || !make_map(&m.dv, dv, 2, d, Nk, BHkv) ||
      !make_map(&m.dqacc, p.ws_dq, 4, d, N, BHq))
    return FA_ERR_CUDA;
  const cudaError_t e = fa::launch_bwd_dkdv(d, m, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

namespace {
// Head dims 136..256: the three passes of fa_bwd_wide.cu after the
// preprocess (no dQ accumulator in the workspace).
fa_status bwd_wide(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                   int N, int Nk, int d, int causal, float scale, void* stream) {
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p{};
  int num_sms = 0;
  fa_status st = bwd_setup(B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes, &p, &num_sms, stream, true,
                           nullptr, 0, 0, Nk);
  if (st != FA_OK) return st;
  fa::BwdMaps m, m64;
  const long long BHq = static_cast<long long>(B) * Hq, BHkv = static_cast<long long>(B) * Hkv;
  if (!make_map(&m.q, q, 2, d, N, BHq) || !make_map(&m.k, k, 2, d, Nk, BHkv) || !make_map(&m.v, v, 2, d, Nk, BHkv) ||
      !make_map(&m.dO, dO, 2, d, N, BHq) || !make_map(&m.dk, dk, 2, d, Nk, BHkv) ||
      !make_map(&m.dv, dv, 2, d, Nk, BHkv) || !make_map(&m.dq, dq, 2, d, N, BHq) ||
      !make_map(&m64.q, q, 2, d, N, BHq, 64) || !make_map(&m64.dO, dO, 2, d, N, BHq, 64) ||
      !make_map(&m64.k, k, 2, d, Nk, BHkv, 64) || !make_map(&m64.v, v, 2, d, Nk, BHkv, 64))
    return FA_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_bwd_pre(d, o, dO, lse, p, num_sms, s);
  if (e == cudaSuccess) e = fa::launch_bwd_wide(m, m64, p, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

extern "C" {

fa_status fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv,
                      void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, int causal,
                      float scale, void* stream) {
  return bwd_dkdv_common(q, k, v, dO, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, N, d, causal, scale,
                         stream);
}

fa_status fa_bwd_dq(void* dq, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d,
                    float scale, void* stream) {
  if (!dq || !aligned16(dq)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p{};
  int num_sms = 0;
  fa_status st = bwd_setup(B, Hq, Hkv, N, d, 0, scale, workspace, workspace_bytes, &p, &num_sms, stream);
  if (st != FA_OK) return st;
  const cudaError_t e = fa::launch_bwd_dq(d, dq, p, num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                 int N, int d, int causal, float scale, void* stream) {
  if (d > 128)
    return bwd_wide(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, N, d, causal, scale,
                    stream);
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  fa_status st = fa_bwd_preprocess(o, lse, dO, workspace, workspace_bytes, B, Hq, Hkv, N, d, stream);
  if (st != FA_OK) return st;
  st = fa_bwd_dkdv(q, k, v, dO, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d, causal, scale, stream);
  if (st != FA_OK) return st;
  return fa_bwd_dq(dq, workspace, workspace_bytes, B, Hq, Hkv, N, d, scale, stream);
}

fa_status fa_bwd_kv(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                    void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                    int Nq, int Nk, int d, int causal, float scale, void* stream) {
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  if (d > 128)
    return bwd_wide(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nk, d, causal,
                    scale, stream);
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  fa_status st = fa_bwd_preprocess(o, lse, dO, workspace, workspace_bytes, B, Hq, Hkv, Nq, d, stream);
  if (st != FA_OK) return st;
  st = bwd_dkdv_common(q, k, v, dO, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, Nq, Nk, d, causal, scale, stream);
  if (st != FA_OK) return st;
  return fa_bwd_dq(dq, workspace, workspace_bytes, B, Hq, Hkv, Nq, d, scale, stream);
}

fa_status fa_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                               const void* dO, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                               int B, int Hq, int Hkv, int N, int d, int causal, float scale, void* stream) {
  if (d > 128)       // the three-pass backward is bit reproducible too
    return bwd_wide(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, N, d, causal, scale,
                    stream);
  const void* ptrs[] = {q, k, v, o, lse, dO, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  fa::BwdParams p{};
  int num_sms = 0;
  fa_status st = bwd_setup(B, Hq, Hkv, N, d, causal, scale, workspace, workspace_bytes, &p, &num_sms, stream, true);
  if (st != FA_OK) return st;
  fa::BwdMaps m;
  const long long BHq = static_cast<long long>(B) * Hq, BHkv = static_cast<long long>(B) * Hkv;
  if (!make_map(&m.q, q, 2, d, N, BHq) || !make_map(&m.k, k, 2, d, N, BHkv) || !make_map(&m.v, v, 2, d, N, BHkv) ||
      !make_map(&m.dO, dO, 2, d, N, BHq) || !make_map(&m.dk, dk, 2, d, N, BHkv) || !make_map(&m.dv, dv, 2, d, N, BHkv) ||
      !make_map(&m.dq, dq, 2, d, N, BHq))
    return FA_ERR_CUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_bwd_pre(d, o, dO, lse, p, num_sms, s);
  if (e == cudaSuccess) e = fa::launch_bwd_deterministic(d, m, p, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                 int d, int causal, float scale, void* stream) {
  return fwd_common(2, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, stream);
}

fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                    int Nk, int d, int causal, float scale, void* stream) {
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  return fwd_common(2, q, k, v, o, lse, B, Hq, Hkv, Nq, d, causal, scale, stream, nullptr, 0, 0, Nk);
}

fa_status fa_fwd_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int Nq, int Nk, int d, int causal, float scale, void* stream) {
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  return fwd_common(2, q, k, v, o, lse, B, Hq, Hkv, Nq, d, causal, scale, stream, nullptr, 0, 0, Nk, true);
}

fa_status fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                             const unsigned char* block_mask, long long mask_stride_b, long long mask_stride_h, int B,
                             int Hq, int Hkv, int N, int d, int causal, float scale, void* stream) {
  if (!block_mask || mask_stride_b < 0 || mask_stride_h < 0) return FA_ERR_INVALID_ARG;
  if ((N + 127) / 128 > fa::kMaskMaxTiles) return FA_ERR_UNSUPPORTED;
  return fwd_common(2, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, stream, block_mask, mask_stride_b,
                    mask_stride_h);
}

fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int Hq, int Hkv,
                     int N, int d, int causal, float scale, void* stream) {
  return fwd_common(4, q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, stream);
}

size_t fa_fp8_row_scales(int N) { return N >= 1 ? static_cast<size_t>((N + 63) / 64) : 0; }

size_t fa_fp8_vt_keys(int N) { return N >= 1 ? static_cast<size_t>((N + 127) / 128 * 128) : 0; }

fa_status fa_fp8_quantize_rows(const void* x, void* out, float* scales, int BH, int N, int d, void* stream) {
  if (!x || !out || !scales || !aligned16(x) || !aligned16(out) || !aligned16(scales)) return FA_ERR_INVALID_ARG;
  if (BH < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (!fp8_dim(d)) return FA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  const fa_status st = device_state(stream, &status);
  if (st != FA_OK) return st;
  return fa::launch_fp8_quant_rows(x, out, scales, BH, N, d, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fp8_quantize_v(const void* v, void* vt, float* scales, int BH, int N, int d, void* stream) {
  if (!v || !vt || !scales || !aligned16(v) || !aligned16(vt) || !aligned16(scales)) return FA_ERR_INVALID_ARG;
  if (BH < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
  if (!fp8_dim(d)) return FA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  const fa_status st = device_state(stream, &status);
  if (st != FA_OK) return st;
  return fa::launch_fp8_quant_v(v, vt, scales, BH, N, d, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"

namespace {
fa_status fwd_fp8_common(const void* q, const float* q_scale, const void* k, const float* k_scale, const void* vt,
                         const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int N, int Nk, int d,
                         int causal, float scale, void* stream) {
  const void* ptrs[] = {q, q_scale, k, k_scale, vt, v_scale, o, lse};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, Hq, Hkv, N, d, scale);
  if (st != FA_OK) return st;
  if (Nk < 1 || check_sizes(B, Hq, Hkv, Nk, d, scale) != FA_OK) return FA_ERR_INVALID_ARG;
  if (!fp8_dim(d)) return FA_ERR_UNSUPPORTED;
  unsigned* status = nullptr;
  st = device_state(stream, &status);
  if (st != FA_OK) return st;
  CUtensorMap mq, mk, mvt, mo;
  const long long BHq = static_cast<long long>(B) * Hq, BHkv = static_cast<long long>(B) * Hkv;
  const int NP = (Nk + 127) / 128 * 128;
  if (!make_map(&mq, q, 1, d, N, BHq) || !make_map(&mk, k, 1, d, Nk, BHkv) ||
      !make_map(&mvt, vt, 1, NP, d, BHkv) || !make_map(&mo, o, 2, d, N, BHq))
    return FA_ERR_CUDA;
  fa::FwdParams p{};
  p.lse = lse;
  p.status = status;
  p.N = N;
  p.Nk = Nk;
  p.causal_off = Nk - N;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.BH = static_cast<int>(BHq);
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = wait_limit_ns();
  p.test_stall = test_stall();
  p.head_dim = d;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d <= 128 ? fa::launch_fwd_fp8(mq, mk, mvt, mo, p, s) : fa::launch_fwd_fp8_wide(mq, mk, mvt, mo, p, s);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

extern "C" {

fa_status fa_fwd_fp8(const void* q, const float* q_scale, const void* k, const float* k_scale, const void* vt,
                     const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int N, int d, int causal,
                     float scale, void* stream) {
  return fwd_fp8_common(q, q_scale, k, k_scale, vt, v_scale, o, lse, B, Hq, Hkv, N, N, d, causal, scale, stream);
}

fa_status fa_fwd_fp8_kv(const void* q, const float* q_scale, const void* k, const float* k_scale, const void* vt,
                        const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                        int causal, float scale, void* stream) {
  return fwd_fp8_common(q, q_scale, k, k_scale, vt, v_scale, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, stream);
}

fa_status fa_ex2_throughput(double* per_sm_per_cycle, void* stream) {
  if (!per_sm_per_cycle) return FA_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  int num_sms = 0;
  const fa_status st = device_state(stream, &status, &num_sms);
  if (st != FA_OK) return st;
  if (num_sms > fa::kEx2MaxSms) return FA_ERR_UNSUPPORTED;
  return fa::measure_ex2_rate(num_sms, 4096, per_sm_per_cycle, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_device_status(void* stream) {
  unsigned* status = nullptr;
  fa_status st = device_state(stream, &status);
  if (st != FA_OK) return st;
  // read and clear this stream's word in the stream's own order: work on
  // other streams is neither waited for nor reported here
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned host = 0;
  if (cudaMemcpyAsync(&host, status, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  if (host != 0) {
    if (cudaMemsetAsync(status, 0, sizeof(unsigned), s) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    return (host & 1u) ? FA_ERR_TIMEOUT : FA_ERR_DEVICE;
  }
  return FA_OK;
}

fa_status fa_sm_clock_mhz(double* mhz, void* stream) {
  if (!mhz) return FA_ERR_INVALID_ARG;
  unsigned* status = nullptr;
  unsigned long long* acc = nullptr;
  const fa_status st = device_state(stream, &status, nullptr, &acc);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  unsigned long long host[2] = {0, 0};
  if (cudaMemcpyAsync(host, acc, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemsetAsync(acc, 0, sizeof(host), s) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
  *mhz = host[1] > 0 ? static_cast<double>(host[0]) * 1e3 / static_cast<double>(host[1]) : 0.0;
  return FA_OK;
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, or bad size)";
    case FA_ERR_UNSUPPORTED: return "unsupported combination of sizes or types";
    case FA_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103)";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out; outputs of that call are invalid";
    case FA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case FA_ERR_DEVICE: return "a kernel refused to run on this device's shared-memory layout; outputs invalid";
  }
  return "unknown status";
}

int fa_version(void) { return 400; }

}  // extern "C"
