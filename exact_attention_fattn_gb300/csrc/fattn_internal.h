// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fattn {

struct DeviceStatus;

// Everything a forward launch needs besides the tensor maps.
struct FwdArgs {
  uint16_t* o;                // bf16 [BH, N, d]
  float* lse;                 // [BH, N]
  DeviceStatus* status;
  long long wait_budget;      // cycles
  int N;
  int BH;
  int sec_heads;              // heads per scheduling section (set by the launcher)
  float scale_log2;           // scale * log2(e)
  float tau_log2;             // rescale threshold (log2 units)
  // FP8 only (nullptr otherwise): block scales [BH, ceil(N/128)] of Q, K, V
  const float* sq;
  const float* sk;
  const float* sv;
};

// Launch the forward kernel for head dim d (64/128).  Tensor maps are 3-D
// {d, N, B*H} views of q, k, v with 128-row boxes and a 128-byte swizzle.
cudaError_t launch_fwd(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdArgs& a, cudaStream_t stream);

// FP8 forward (d = 128): tq, tk are 3-D uint8 views {d, N, B*H} of the e4m3
// codes with 128-byte x 128-row boxes; tv a 3-D uint8 view {Np, d, B*H} of the
// transposed V codes with the same box.
cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const FwdArgs& a, cudaStream_t stream);

// Block quantization to e4m3: one scale per 128 rows of a head (amax / 448),
// codes [BH, N, d] or, transposed, [BH, d, Np] with zero codes past N.
cudaError_t launch_fp8_quantize(const void* x, void* codes, float* scales, int BH, int N, int d,
                                bool transpose, cudaStream_t stream);

// The same after the randomized Hadamard rotation diag(signs) H / sqrt(d) of
// every row (d = 128; not transposed).
cudaError_t launch_fp8_quantize_rotated(const void* x, const float* signs, void* codes,
                                        float* scales, int BH, int N, int d,
                                        cudaStream_t stream);

// Capacity of the backward's tail tables (kernel parameters, ~2.6 KB).
constexpr int kBwdTailMaxCtas = 256;
constexpr int kBwdTailCap = 1024;

struct BwdArgs {
  const float* L2;            // [BH, Np]: -lse * log2(e), -inf past N (Np = N rounded up to 128)
  const float* D;             // [BH, Np]: rowsum(dO o O), 0 past N
  float* dq_accum;            // [BH, N, d] fp32
  uint32_t* dq_order;         // [BH, n_tiles] contribution counters, or nullptr (any order)
  uint16_t* dk;               // bf16 [BH, N, d]
  uint16_t* dv;               // bf16 [BH, N, d]
  DeviceStatus* status;
  long long wait_budget;
  int N;
  int BH;
  int sec_heads;              // heads per scheduling section (set by the launcher)
  int paired;                 // causal K/V tiles p and n - 1 - p paired (set by the launcher)
  float scale;
  float scale_log2;
  // Paired causal schedule only (set by the launcher, see bwd_item): the
  // last tail_heads heads are dealt K/V tile by K/V tile from these tables.
  int tail_heads;
  uint16_t tail_off[kBwdTailMaxCtas + 1];  // CTA c: entries [tail_off[c], tail_off[c + 1])
  uint16_t tail_item[kBwdTailCap];         // r * n_tiles + j: K/V tile j of head BH - tail_heads + r
};

// D (and, when L2 != nullptr, L2 = -lse * log2 e) in a [BH, pitch] layout with
// padding rows N..pitch-1; zeroes dq_accum [BH, N, d] and, when given, the
// [BH, pitch / 128] dQ contribution counters.
cudaError_t launch_bwd_preprocess(const void* o, const void* dO, const float* lse, float* D,
                                  float* L2, float* dq_accum, uint32_t* counters, int BH, int N,
                                  int pitch, int d, cudaStream_t stream);

// tacc: 3-D fp32 view {d, N, B*H} of the dQ accumulator, 32 x 32 boxes,
// 128-byte swizzle (the target of the dQ reduce-adds).
cudaError_t launch_bwd_main(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tacc, const BwdArgs& a, cudaStream_t stream);

// CTA-pair version of the main backward kernel (d = 128, any-order dQ; see
// fattn_bwd2.cu).  tq64 / tdo64: views of q and dO with 64-row boxes.
cudaError_t launch_bwd2_main(bool causal, const CUtensorMap& tq, const CUtensorMap& tq64,
                             const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                             const CUtensorMap& tdo64, const CUtensorMap& tacc, const BwdArgs& a,
                             cudaStream_t stream);

cudaError_t launch_dq_convert(const float* dq_accum, void* dq, long long elems, float scale,
                              cudaStream_t stream);

cudaError_t launch_selftest_timeout(DeviceStatus* status, long long budget, cudaStream_t stream);

}  // namespace fattn
