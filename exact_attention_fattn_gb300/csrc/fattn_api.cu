// C-ABI boundary of libfattn: argument validation, tensor-map construction,
// launch sequencing and the device status word.  See include/fattn.h.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/fattn.h"
#include "fattn_internal.h"
#include "fattn_ptx.cuh"
#include "fattn_sched.h"

namespace fattn {

// An NVTX range around each entry point that enqueues work, so that
// profiler timelines show the library's calls (no cost without a tool).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// The single status word of the library on each device.
__device__ DeviceStatus g_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultBudget = 1ll << 31;

std::mutex g_mu;
DeviceStatus* g_status_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 unsupported
long long g_budget = kDefaultBudget;
float g_tau_log2 = 8.0f;
constexpr float kFp8TauMax = 8.0f;
bool g_deterministic = false;
bool g_bwd_pair = false;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device setup: architecture check and the status word's address.
int device_setup(DeviceStatus** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FATTN_ERR_CUDA;
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_arch_ok[dev] < 0) return FATTN_ERR_UNSUPPORTED;
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return FATTN_ERR_CUDA;
    g_status_ptr[dev] = static_cast<DeviceStatus*>(p);
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return FATTN_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *status = g_status_ptr[dev];
  return FATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_sizes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0) return FATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FATTN_ERR_UNSUPPORTED;
  const long long elems = static_cast<long long>(B) * H * N * d;
  if (elems >= (1ll << 31)) return FATTN_ERR_INVALID_ARG;
  return FATTN_OK;
}

bool scale_ok(float s) { return isfinite(s) && s > 0.f; }

// 3-D bf16 view {d, N, B*H} of a [B,H,N,d] tensor, 64-column x box_rows boxes,
// 128-byte swizzle, zero fill outside the tensor.
int make_map(CUtensorMap* m, const void* ptr, int N, int BH, int d, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FATTN_OK : FATTN_ERR_CUDA;
}

// 3-D uint8 view {inner, rows, B*H} of e4m3 codes, 128-byte x 128-row boxes,
// 128-byte swizzle, zero fill outside the tensor.
int make_map_u8(CUtensorMap* m, const void* ptr, int inner, int rows, int BH) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                                 static_cast<cuuint64_t>(rows) * inner};
  const cuuint32_t box[3] = {128u, 128u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FATTN_OK : FATTN_ERR_CUDA;
}

// 3-D fp32 view {d, N, B*H} of the dQ accumulator: 32-column (128-byte) x
// 32-row boxes, 128-byte swizzle.
int make_acc_map(CUtensorMap* m, const void* ptr, int N, int BH, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(N) * d * 4};
  const cuuint32_t box[3] = {32u, 32u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FATTN_OK : FATTN_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? FATTN_OK : FATTN_ERR_CUDA; }

}  // namespace
}  // namespace fattn

using namespace fattn;

extern "C" {

int fattn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int N, int d, int causal, float scale, fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_fwd");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (!q || !k || !v || !o || !lse) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if ((rc = make_map(&tq, q, N, BH, d, 128)) != FATTN_OK) return rc;
  if ((rc = make_map(&tk, k, N, BH, d, 128)) != FATTN_OK) return rc;
  if ((rc = make_map(&tv, v, N, BH, d, 128)) != FATTN_OK) return rc;
  FwdArgs a;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.status = status;
  a.N = N;
  a.BH = BH;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.sq = a.sk = a.sv = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.wait_budget = g_budget;
    a.tau_log2 = g_tau_log2;
  }
  return from_cuda(launch_fwd(d, causal != 0, tq, tk, tv, a,
                              reinterpret_cast<cudaStream_t>(stream)));
}

size_t fattn_fp8_codes_bytes(int B, int H, int N, int d, int transposed) {
  if (check_sizes(B, H, N, d) != FATTN_OK || d != 128) return 0;
  const size_t rows = transposed ? static_cast<size_t>(N + 127) / 128 * 128 : N;
  return static_cast<size_t>(B) * H * rows * d;
}

int fattn_quantize_fp8(const void* x, void* codes, float* scales, int B, int H, int N, int d,
                       int transposed, fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_quantize_fp8");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (d != 128) return FATTN_ERR_UNSUPPORTED;
  if (!x || !codes || !scales) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  return from_cuda(launch_fp8_quantize(x, codes, scales, B * H, N, d, transposed != 0,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int fattn_quantize_fp8_rotated(const void* x, const float* signs, void* codes, float* scales,
                               int B, int H, int N, int d, fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_quantize_fp8_rotated");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (d != 128) return FATTN_ERR_UNSUPPORTED;
  if (!x || !signs || !codes || !scales) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(signs) || !aligned16(codes) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  return from_cuda(launch_fp8_quantize_rotated(x, signs, codes, scales, B * H, N, d,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

int fattn_fwd_fp8(const void* q8, const float* sq, const void* k8, const float* sk,
                  const void* v8t, const float* sv, void* o, float* lse, int B, int H, int N,
                  int d, int causal, float scale, fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_fwd_fp8");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (d != 128) return FATTN_ERR_UNSUPPORTED;
  if (!q8 || !sq || !k8 || !sk || !v8t || !sv || !o || !lse) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(o) || !aligned16(lse))
    return FATTN_ERR_INVALID_ARG;
  for (const float* p : {sq, sk, sv})
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0) return FATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  const int BH = B * H;
  const int np = (N + 127) / 128 * 128;
  CUtensorMap tq, tk, tv;
  if ((rc = make_map_u8(&tq, q8, d, N, BH)) != FATTN_OK) return rc;
  if ((rc = make_map_u8(&tk, k8, d, N, BH)) != FATTN_OK) return rc;
  if ((rc = make_map_u8(&tv, v8t, np, d, BH)) != FATTN_OK) return rc;
  FwdArgs a;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.status = status;
  a.N = N;
  a.BH = BH;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.wait_budget = g_budget;
    // The e4m3 probabilities P * rho reach 2^tau (rho <= 1); e4m3 saturates
    // at 448 = 2^8.81, so the FP8 forward never lets tau above 8.
    a.tau_log2 = g_tau_log2 > kFp8TauMax ? kFp8TauMax : g_tau_log2;
  }
  return from_cuda(launch_fwd_fp8(causal != 0, tq, tk, tv, a,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

// Workspace of the backward pass: D and -L*log2(e) in a [B*H, Np] layout
// (Np = N rounded up to the 128-row tile, so that every tile's 512-byte
// slice can be fetched by one bulk copy), then the fp32 dQ accumulator, then
// one uint32 dQ contribution counter per (head, 128-row Q tile).
}  // extern "C"
namespace {
struct BwdWorkspace {
  size_t d_off, l2_off, acc_off, cnt_off, total;
  int pitch;
};

BwdWorkspace bwd_workspace(int B, int H, int N, int d) {
  BwdWorkspace w;
  w.pitch = (N + 127) / 128 * 128;
  const size_t prow = static_cast<size_t>(B) * H * w.pitch;
  const size_t rows = static_cast<size_t>(B) * H * N;
  w.d_off = 0;
  w.l2_off = align256(prow * sizeof(float));
  w.acc_off = w.l2_off + align256(prow * sizeof(float));
  w.cnt_off = w.acc_off + align256(rows * d * sizeof(float));
  w.total = w.cnt_off + align256(static_cast<size_t>(B) * H * (w.pitch / 128) * sizeof(uint32_t));
  return w;
}
}  // namespace
extern "C" {

size_t fattn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d) != FATTN_OK) return 0;
  return bwd_workspace(B, H, N, d).total;
}

int fattn_bwd_preprocess(const void* o, const void* dO, float* D, float* dq_accum, int B, int H,
                         int N, int d, fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_bwd_preprocess");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (!o || !dO || !D || !dq_accum) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(D) || !aligned16(dq_accum))
    return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  return from_cuda(launch_bwd_preprocess(o, dO, nullptr, D, nullptr, dq_accum, nullptr, B * H,
                                         N, N, d, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

int check_workspace(const void* workspace, size_t workspace_bytes, int B, int H, int N, int d) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FATTN_ERR_INVALID_ARG;
  if (workspace_bytes < bwd_workspace(B, H, N, d).total) return FATTN_ERR_INVALID_ARG;
  return FATTN_OK;
}

int bwd_prepare_impl(const void* o, const void* dO, const float* lse, void* workspace, int B,
                     int H, int N, int d, cudaStream_t st) {
  const BwdWorkspace ws = bwd_workspace(B, H, N, d);
  char* wbase = static_cast<char*>(workspace);
  return from_cuda(launch_bwd_preprocess(
      o, dO, lse, reinterpret_cast<float*>(wbase + ws.d_off),
      reinterpret_cast<float*>(wbase + ws.l2_off), reinterpret_cast<float*>(wbase + ws.acc_off),
      reinterpret_cast<uint32_t*>(wbase + ws.cnt_off), B * H, N, ws.pitch, d, st));
}

int bwd_main_impl(const void* q, const void* k, const void* v, const void* dO, void* workspace,
                  void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                  DeviceStatus* status, cudaStream_t st) {
  const int BH = B * H;
  const BwdWorkspace ws = bwd_workspace(B, H, N, d);
  char* wbase = static_cast<char*>(workspace);
  int rc;
  CUtensorMap tq, tk, tv, tdo, tacc;
  if ((rc = make_map(&tq, q, N, BH, d, 128)) != FATTN_OK) return rc;
  if ((rc = make_map(&tk, k, N, BH, d, 128)) != FATTN_OK) return rc;
  if ((rc = make_map(&tv, v, N, BH, d, 128)) != FATTN_OK) return rc;
  if ((rc = make_map(&tdo, dO, N, BH, d, 128)) != FATTN_OK) return rc;
  if ((rc = make_acc_map(&tacc, wbase + ws.acc_off, N, BH, d)) != FATTN_OK) return rc;
  bool pair = false;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    pair = g_bwd_pair && !g_deterministic && d == 128;
  }
  BwdArgs a;
  a.L2 = reinterpret_cast<const float*>(wbase + ws.l2_off);
  a.D = reinterpret_cast<const float*>(wbase + ws.d_off);
  a.dq_accum = reinterpret_cast<float*>(wbase + ws.acc_off);
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.status = status;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    a.wait_budget = g_budget;
    a.dq_order = g_deterministic ? reinterpret_cast<uint32_t*>(wbase + ws.cnt_off) : nullptr;
  }
  a.N = N;
  a.BH = BH;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  if (pair) {
    CUtensorMap tq64, tdo64;
    if ((rc = make_map(&tq64, q, N, BH, d, 64)) != FATTN_OK) return rc;
    if ((rc = make_map(&tdo64, dO, N, BH, d, 64)) != FATTN_OK) return rc;
    return from_cuda(launch_bwd2_main(causal != 0, tq, tq64, tk, tv, tdo, tdo64, tacc, a, st));
  }
  return from_cuda(launch_bwd_main(d, causal != 0, tq, tk, tv, tdo, tacc, a, st));
}

int bwd_finish_impl(const void* workspace, void* dq, int B, int H, int N, int d, float scale,
                    cudaStream_t st) {
  const BwdWorkspace ws = bwd_workspace(B, H, N, d);
  const float* acc =
      reinterpret_cast<const float*>(static_cast<const char*>(workspace) + ws.acc_off);
  return from_cuda(
      launch_dq_convert(acc, dq, static_cast<long long>(B) * H * N * d, scale, st));
}

}  // namespace

extern "C" {

int fattn_bwd_prepare(const void* o, const void* dO, const float* lse, void* workspace,
                      size_t workspace_bytes, int B, int H, int N, int d,
                      fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_bwd_prepare");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (!o || !dO || !lse) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(lse)) return FATTN_ERR_INVALID_ARG;
  if ((rc = check_workspace(workspace, workspace_bytes, B, H, N, d)) != FATTN_OK) return rc;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  return bwd_prepare_impl(o, dO, lse, workspace, B, H, N, d,
                          reinterpret_cast<cudaStream_t>(stream));
}

int fattn_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* workspace,
                   size_t workspace_bytes, void* dk, void* dv, int B, int H, int N, int d,
                   int causal, float scale, fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_bwd_main");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (!q || !k || !v || !dO || !dk || !dv) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dk) ||
      !aligned16(dv))
    return FATTN_ERR_INVALID_ARG;
  if ((rc = check_workspace(workspace, workspace_bytes, B, H, N, d)) != FATTN_OK) return rc;
  if (!scale_ok(scale)) return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  return bwd_main_impl(q, k, v, dO, workspace, dk, dv, B, H, N, d, causal, scale, status,
                       reinterpret_cast<cudaStream_t>(stream));
}

int fattn_bwd_finish(const void* workspace, size_t workspace_bytes, void* dq, int B, int H, int N,
                     int d, float scale, fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_bwd_finish");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (!dq || !aligned16(dq)) return FATTN_ERR_INVALID_ARG;
  if ((rc = check_workspace(workspace, workspace_bytes, B, H, N, d)) != FATTN_OK) return rc;
  if (!scale_ok(scale)) return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  return bwd_finish_impl(workspace, dq, B, H, N, d, scale, reinterpret_cast<cudaStream_t>(stream));
}

int fattn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
              const float* lse, void* dq, void* dk, void* dv, void* workspace,
              size_t workspace_bytes, int B, int H, int N, int d, int causal, float scale,
              fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_bwd");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FATTN_ERR_INVALID_ARG;
  if ((rc = check_workspace(workspace, workspace_bytes, B, H, N, d)) != FATTN_OK) return rc;
  if (!scale_ok(scale)) return FATTN_ERR_INVALID_ARG;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = bwd_prepare_impl(o, dO, lse, workspace, B, H, N, d, st)) != FATTN_OK) return rc;
  if ((rc = bwd_main_impl(q, k, v, dO, workspace, dk, dv, B, H, N, d, causal, scale, status,
                          st)) != FATTN_OK)
    return rc;
  return bwd_finish_impl(workspace, dq, B, H, N, d, scale, st);
}

int fattn_bwd_schedule(int B, int H, int N, int d, int causal, int deterministic, int grid,
                       long long l2_bytes, int* item_cta, long long* cta_q_tiles) {
  const int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (grid <= 0 || l2_bytes < 0 || !item_cta) return FATTN_ERR_INVALID_ARG;
  const int BH = B * H;
  const int n_tiles = (N + 127) / 128;
  const long long items = static_cast<long long>(n_tiles) * BH;
  if (items > (1ll << 24) || grid > items) return FATTN_ERR_INVALID_ARG;
  BwdArgs a{};
  a.N = N;
  a.BH = BH;
  // The item function only tests the counter pointer against null.
  uint32_t dummy_order = 0;
  a.dq_order = deterministic ? &dummy_order : nullptr;
  plan_bwd_schedule(a, n_tiles, d, causal != 0, deterministic != 0, grid, l2_bytes);
  for (long long i = 0; i < items; ++i) item_cta[i] = -1;
  for (int c = 0; c < grid; ++c) {
    long long walked = 0;
    BwdItem w;
    for (int m = 0; m <= items; ++m) {
      const bool more = causal ? bwd_item<true>(m, n_tiles, a, grid, c, w)
                               : bwd_item<false>(m, n_tiles, a, grid, c, w);
      if (!more) break;
      int& slot = item_cta[static_cast<long long>(w.bh) * n_tiles + w.j];
      slot = slot == -1 ? c : -2;
      walked += w.n_it;
    }
    if (cta_q_tiles) cta_q_tiles[c] = walked;
  }
  return FATTN_OK;
}

int fattn_bwd_schedule_items(int B, int H, int N, int d, int causal, int deterministic, int grid,
                             long long l2_bytes, int* cta_start, int* items) {
  const int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (grid <= 0 || l2_bytes < 0 || !cta_start || !items) return FATTN_ERR_INVALID_ARG;
  const int BH = B * H;
  const int n_tiles = (N + 127) / 128;
  const long long n_items = static_cast<long long>(n_tiles) * BH;
  if (n_items > (1ll << 24) || grid > n_items) return FATTN_ERR_INVALID_ARG;
  BwdArgs a{};
  a.N = N;
  a.BH = BH;
  uint32_t dummy_order = 0;
  a.dq_order = deterministic ? &dummy_order : nullptr;
  plan_bwd_schedule(a, n_tiles, d, causal != 0, deterministic != 0, grid, l2_bytes);
  long long e = 0;
  for (int c = 0; c < grid; ++c) {
    cta_start[c] = static_cast<int>(e);
    BwdItem w;
    for (int m = 0; m <= n_items; ++m) {
      const bool more = causal ? bwd_item<true>(m, n_tiles, a, grid, c, w)
                               : bwd_item<false>(m, n_tiles, a, grid, c, w);
      if (!more) break;
      if (e >= n_items) return FATTN_ERR_INVALID_ARG;   // more entries than items: not a schedule
      int* out = items + 5 * e;
      out[0] = w.bh;
      out[1] = w.j;
      out[2] = w.i0;
      out[3] = w.n_it;
      out[4] = w.rot;
      ++e;
    }
  }
  cta_start[grid] = static_cast<int>(e);
  return FATTN_OK;
}

int fattn_bwd_pair_schedule_items(int B, int H, int N, int causal, int clusters,
                                  long long l2_bytes, int* cluster_start, int* items) {
  const int rc = check_sizes(B, H, N, 128);
  if (rc != FATTN_OK) return rc;
  if (clusters <= 0 || l2_bytes < 0 || !cluster_start || !items) return FATTN_ERR_INVALID_ARG;
  const int BH = B * H;
  const int n_tiles = (N + 127) / 128;
  const long long n_units = static_cast<long long>((n_tiles + 1) / 2) * BH;
  if (n_units > (1ll << 24) || clusters > n_units) return FATTN_ERR_INVALID_ARG;
  BwdArgs a{};
  a.N = N;
  a.BH = BH;
  plan_bwd2_schedule(a, n_tiles, causal != 0, clusters, l2_bytes);
  long long e = 0;
  for (int c = 0; c < clusters; ++c) {
    cluster_start[c] = static_cast<int>(e);
    BwdItem w;
    for (int m = 0; m <= n_units; ++m) {
      const bool more = causal ? bwd2_item<true>(m, n_tiles, a, clusters, c, w)
                               : bwd2_item<false>(m, n_tiles, a, clusters, c, w);
      if (!more) break;
      if (e >= n_units) return FATTN_ERR_INVALID_ARG;   // more entries than units: not a schedule
      int* out = items + 5 * e;
      out[0] = w.bh;
      out[1] = w.j;
      out[2] = w.i0;
      out[3] = w.n_it;
      out[4] = w.rot;
      ++e;
    }
  }
  cluster_start[clusters] = static_cast<int>(e);
  return FATTN_OK;
}

int fattn_check_status(fattn_stream_t stream) {
  const NvtxRange nvtx_range("fattn_check_status");
  DeviceStatus* status = nullptr;
  int rc = device_setup(&status);
  if (rc != FATTN_OK) return rc;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FATTN_ERR_CUDA;
  e = cudaGetLastError();
  if (e != cudaSuccess) return FATTN_ERR_CUDA;
  DeviceStatus host = {};
  if (cudaMemcpyFromSymbol(&host, g_status, sizeof(host)) != cudaSuccess) return FATTN_ERR_CUDA;
  if (host.code != 0) {
    DeviceStatus zero = {};
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return FATTN_ERR_CUDA;
    return static_cast<int>(host.code);
  }
  return FATTN_OK;
}

const char* fattn_status_string(int status) {
  switch (status) {
    case FATTN_OK: return "ok";
    case FATTN_ERR_INVALID_ARG: return "invalid argument";
    case FATTN_ERR_UNSUPPORTED: return "unsupported head dimension or device";
    case FATTN_ERR_CUDA: return "CUDA error";
    case FATTN_ERR_TIMEOUT: return "kernel wait timed out";
    case FATTN_ERR_TOO_LARGE: return "problem exceeds the built-in scratch of fattn_bwd_noalloc";
    case FATTN_ERR_DEBUG_CHECK: return "a debug-build range check failed in a kernel";
    default: return "unknown status";
  }
}

void fattn_set_wait_budget(long long cycles) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_budget = cycles > 0 ? cycles : kDefaultBudget;
}

void fattn_set_deterministic(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_deterministic = on != 0;
}

void fattn_set_bwd_pair(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_bwd_pair = on != 0;
}

void fattn_set_rescale_threshold(float tau_log2) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!(tau_log2 >= 0.f)) tau_log2 = 8.0f;
  g_tau_log2 = tau_log2 > 16.f ? 16.f : tau_log2;
}

int fattn_selftest_timeout(long long budget_cycles, fattn_stream_t stream) {
  DeviceStatus* status = nullptr;
  int rc = device_setup(&status);
  if (rc != FATTN_OK) return rc;
  if (budget_cycles <= 0) return FATTN_ERR_INVALID_ARG;
  return from_cuda(
      launch_selftest_timeout(status, budget_cycles, reinterpret_cast<cudaStream_t>(stream)));
}

const char* fattn_version(void) { return "0.1.0"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward pass without allocation: its scratch lives in this fixed device
// array.  In host code the name is only a stand-in for the symbol; the
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_fattn_noalloc_scratch[FATTN_NOALLOC_SCRATCH_BYTES];

namespace fattn {
namespace {
void* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace
}  // namespace fattn

extern "C" int fattn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                 const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                 int B, int H, int N, int d, int causal, float scale,
                                 fattn_stream_t stream) {
  const fattn::NvtxRange nvtx_range("fattn_bwd_noalloc");
  int rc = check_sizes(B, H, N, d);
  if (rc != FATTN_OK) return rc;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FATTN_ERR_INVALID_ARG;
  if (bwd_workspace(B, H, N, d).total > FATTN_NOALLOC_SCRATCH_BYTES) return FATTN_ERR_TOO_LARGE;
  DeviceStatus* status = nullptr;
  if ((rc = device_setup(&status)) != FATTN_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FATTN_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_fattn_noalloc_scratch) != cudaSuccess || p == nullptr)
        return FATTN_ERR_CUDA;
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // prepare rewrites D, -L*log2(e) (padding included) and zeroes the dQ
  // accumulator, so nothing depends on what the previous call left behind.
  if ((rc = bwd_prepare_impl(o, dO, lse, scratch, B, H, N, d, st)) != FATTN_OK) return rc;
  if ((rc = bwd_main_impl(q, k, v, dO, scratch, dk, dv, B, H, N, d, causal, scale, status, st)) !=
      FATTN_OK)
    return rc;
  return bwd_finish_impl(scratch, dq, B, H, N, d, scale, st);
}
