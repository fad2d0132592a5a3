// Block quantization of bf16 [B,H,N,d] tensors to e4m3 for the FP8 forward
// ("FlashAttention v1～v4" v3 §3: one scale per computation block instead of
// one per tensor).  A block is 128 consecutive rows of one (batch, head):
//   scale = amax(|x| over the block) / 448 (1 for an all-zero block),
//   code  = e4m3(x * (1 / scale)), round to nearest even, saturating,
// the division, reciprocal and product each rounded to fp32.  V is written
// transposed ([B*H, d, Np], Np = N rounded up to 128, zero codes past N) so
// that the second GEMM of the forward reads it K-major.
#include "fattn_internal.h"
#include "fattn_ptx.cuh"

namespace fattn {

namespace {

constexpr int kQThreads = 256;

template <int HD>
__global__ void __launch_bounds__(kQThreads) quantize_kernel(const uint4* __restrict__ x,
                                                             uint8_t* __restrict__ codes,
                                                             float* __restrict__ scales, int N,
                                                             int n_tiles, bool transpose) {
  constexpr int kVecs = HD / 8;                       // 8 bf16 per 16-byte load
  __shared__ float red[kQThreads / 32];
  __shared__ __align__(16) uint8_t tile[128 * HD];    // transposition staging
  const int bh = blockIdx.x / n_tiles;
  const int t = blockIdx.x - bh * n_tiles;
  const int row0 = t * 128;
  const int rows = min(128, N - row0);
  const uint4* xb = x + (static_cast<size_t>(bh) * N + row0) * kVecs;

  float amax = 0.f;
  for (int i = threadIdx.x; i < rows * kVecs; i += kQThreads) {
    const uint4 v = __ldg(&xb[i]);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const float inv = __fdiv_rn(1.f, s);
  if (threadIdx.x == 0) scales[blockIdx.x] = s;

  for (int i = threadIdx.x; i < 128 * kVecs; i += kQThreads) {
    const int r = i / kVecs;
    uint2 out = make_uint2(0u, 0u);
    if (r < rows) {
      const uint4 v = __ldg(&xb[i]);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
      float f[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 p = __bfloat1622float2(h[k]);
        f[2 * k] = __fmul_rn(p.x, inv);
        f[2 * k + 1] = __fmul_rn(p.y, inv);
      }
      out.x = pack_e4m3x4(f[0], f[1], f[2], f[3]);
      out.y = pack_e4m3x4(f[4], f[5], f[6], f[7]);
    }
    if (transpose) {
      *reinterpret_cast<uint2*>(tile + i * 8) = out;
    } else if (r < rows) {
      *reinterpret_cast<uint2*>(codes + (static_cast<size_t>(bh) * N + row0) * HD + i * 8) = out;
    }
  }
  if (transpose) {
    __syncthreads();
    const size_t np = static_cast<size_t>(n_tiles) * 128;
    // 16 consecutive rows of one column per thread: one 16-byte store
    for (int i = threadIdx.x; i < HD * 8; i += kQThreads) {
      const int col = i >> 3;
      const int r16 = (i & 7) * 16;
      uint32_t w4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v |= static_cast<uint32_t>(tile[(r16 + 4 * q + k) * HD + col]) << (8 * k);
        w4[q] = v;
      }
      *reinterpret_cast<uint4*>(codes + (static_cast<size_t>(bh) * HD + col) * np + row0 + r16) =
          make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
  }
}

}  // namespace

cudaError_t launch_fp8_quantize(const void* x, void* codes, float* scales, int BH, int N, int d,
                                bool transpose, cudaStream_t stream) {
  if (d != 128) return cudaErrorInvalidValue;
  const int n_tiles = (N + 127) / 128;
  const long long blocks = static_cast<long long>(BH) * n_tiles;
  quantize_kernel<128><<<static_cast<unsigned>(blocks), kQThreads, 0, stream>>>(
      static_cast<const uint4*>(x), static_cast<uint8_t*>(codes), scales, N, n_tiles, transpose);
  return cudaGetLastError();
}

}  // namespace fattn
