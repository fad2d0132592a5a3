// Bandwidth-bound helpers of the backward pass, and the timeout self-test.
//
//  preprocess: D_i = sum_k dO_ik O_ik ("6.1 FlashAttention V1详解" §6.1,
//              the identity rowsum(dP o P) = rowsum(dO o O)), and zero the
//              fp32 dQ accumulator and the dQ contribution counters.
//  dq convert: dq = bf16(scale * dq_accum) (the scale of dQ = scale dS K is
//              applied once here instead of on every partial sum).
#include "fattn_internal.h"
#include "fattn_ptx.cuh"

namespace fattn {

namespace {

constexpr int kAuxThreads = 256;

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b) {
  const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 fa = __bfloat1622float2(pa[i]);
    const float2 fb = __bfloat1622float2(pb[i]);
    s = fmaf(fa.x, fb.x, s);
    s = fmaf(fa.y, fb.y, s);
  }
  return s;
}

// One group of HD/8 threads per row; each thread reads 16 bytes of O and dO
// and zeroes 32 bytes of the accumulator row.  Rows are walked in a padded
// index space of `pitch` rows per head: row n < N of head bh gets
//   D[bh*pitch + n]  = sum_k dO O,
//   L2[bh*pitch + n] = -lse[bh*N + n] * log2(e)      (when L2 is given),
// and the padding rows n >= N get D = 0 and L2 = -inf (a column that no
// probability can reach: 2^(s*scale*log2e - inf) = 0).  The first row of
// every 128-row tile also zeroes that tile's counter (pitch is a multiple of
// 128 whenever counters are given).
template <int HD>
__global__ void __launch_bounds__(kAuxThreads) preprocess_kernel(
    const uint4* __restrict__ o, const uint4* __restrict__ dO, const float* __restrict__ lse,
    float* __restrict__ D, float* __restrict__ L2, float4* __restrict__ dq_accum,
    uint32_t* __restrict__ counters, int N, int pitch, long long padded_rows) {
  constexpr int kTpr = HD / 8;          // threads per row
  constexpr int kRowsPerWarp = 32 / kTpr;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kTpr;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * kAuxThreads + threadIdx.x) >> 5;
  const long long num_warps = static_cast<long long>(gridDim.x) * (kAuxThreads / 32);
  // The loop bound is uniform across the warp, so every lane reaches the
  // shuffles; lanes past the last row contribute zeros and store nothing.
  for (long long wrow = warp_id * kRowsPerWarp; wrow < padded_rows;
       wrow += num_warps * kRowsPerWarp) {
    const long long prow = wrow + lane / kTpr;
    const long long bh = prow / pitch;
    const int n = static_cast<int>(prow - bh * pitch);
    const bool in_range = prow < padded_rows;
    const bool valid = in_range && n < N;
    const long long row = bh * N + n;
    const long long idx = row * kTpr + sub;
    float s = valid ? dot8_bf16(__ldg(&o[idx]), __ldg(&dO[idx])) : 0.f;
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (in_range && sub == 0) {
      if (counters != nullptr && (n & 127) == 0) counters[bh * (pitch >> 7) + (n >> 7)] = 0u;
      D[prow] = s;
      if (L2 != nullptr) L2[prow] = valid ? -__ldg(&lse[row]) * 1.4426950408889634f : -INFINITY;
    }
    if (valid) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      dq_accum[2 * idx] = z;
      dq_accum[2 * idx + 1] = z;
    }
  }
}

__global__ void __launch_bounds__(kAuxThreads) dq_convert_kernel(const float4* __restrict__ acc,
                                                                 uint2* __restrict__ out,
                                                                 long long n4, float scale) {
  const long long stride = static_cast<long long>(gridDim.x) * kAuxThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kAuxThreads + threadIdx.x; i < n4;
       i += stride) {
    const float4 a = __ldg(&acc[i]);
    uint2 r;
    r.x = pack_bf16x2(a.x * scale, a.y * scale);
    r.y = pack_bf16x2(a.z * scale, a.w * scale);
    out[i] = r;
  }
}

// Waits on a barrier that nothing completes; the bounded wait must give up.
__global__ void selftest_timeout_kernel(DeviceStatus* status, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{budget, reinterpret_cast<volatile uint32_t*>(&abort_flag), status};
    mbar_wait(smem_u32(&bar), 0, wc, kWaitSelfTest);
  }
  __syncthreads();
}

int grid_for(long long work_items) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long blocks = (work_items + kAuxThreads - 1) / kAuxThreads;
  const long long cap = static_cast<long long>(sms) * 8;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, const void* dO, const float* lse, float* D,
                                  float* L2, float* dq_accum, uint32_t* counters, int BH, int N,
                                  int pitch, int d, cudaStream_t stream) {
  const long long padded_rows = static_cast<long long>(BH) * pitch;
  const int grid = grid_for(padded_rows * (d / 8));
  if (d == 64) {
    preprocess_kernel<64><<<grid, kAuxThreads, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dO), lse, D, L2,
        reinterpret_cast<float4*>(dq_accum), counters, N, pitch, padded_rows);
  } else {
    preprocess_kernel<128><<<grid, kAuxThreads, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dO), lse, D, L2,
        reinterpret_cast<float4*>(dq_accum), counters, N, pitch, padded_rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* dq_accum, void* dq, long long elems, float scale,
                              cudaStream_t stream) {
  const long long n4 = elems / 4;
  dq_convert_kernel<<<grid_for(n4), kAuxThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_accum), static_cast<uint2*>(dq), n4, scale);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(DeviceStatus* status, long long budget, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, budget);
  return cudaGetLastError();
}

}  // namespace fattn
