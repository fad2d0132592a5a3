// Microbenchmark: base-2 exponentials per clock per SM, hardware (MUFU
// ex2.approx) against a cubic polynomial on the FMA pipe, and mixes of the
// two, alone and followed by the bf16 packing the attention kernels apply to
// every probability.  Also checks the polynomial's relative error on the
// device over x in [-130, 1].
//
// The polynomial ("FlashAttention v1～v4" v4 §2: 2^x = 2^floor * 2^frac,
// integer part through the exponent field, fraction by Horner): here
// n = rint(x) by adding and subtracting 1.5 * 2^23, f = x - n in [-1/2, 1/2],
// 2^f ~ c0 + f (c1 + f (c2 + f c3)) with coefficients from a near-minimax
// relative-error fit (see run.py), and 2^n added into the exponent field.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <vector>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ float ex2_hw(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

constexpr float kC0 = 0.9999281167984009f;
constexpr float kC1 = 0.6932609677314758f;
constexpr float kC2 = 0.24261054396629333f;
constexpr float kC3 = 0.05517132207751274f;

// Two elements at a time (packed fp32 pairs).  Inputs below -126.5 are
// clamped there (the result is then a denormal of at most 5e-39).
__device__ __forceinline__ void exp2_poly2(float x0, float x1, float& y0, float& y1) {
  x0 = fmaxf(x0, -126.5f);
  x1 = fmaxf(x1, -126.5f);
  const uint64_t m = pk2(12582912.f, 12582912.f);
  const uint64_t t = add2(pk2(x0, x1), m);
  const uint64_t f = sub2(pk2(x0, x1), sub2(t, m));
  uint64_t p = fma2(pk2(kC3, kC3), f, pk2(kC2, kC2));
  p = fma2(p, f, pk2(kC1, kC1));
  p = fma2(p, f, pk2(kC0, kC0));
  float p0, p1, t0, t1;
  up2(p, p0, p1);
  up2(t, t0, t1);
  y0 = __uint_as_float(__float_as_uint(p0) + (__float_as_uint(t0) << 23));
  y1 = __uint_as_float(__float_as_uint(p1) + (__float_as_uint(t1) << 23));
}

// Sixteen independent chains per thread; NPOLY of them use the polynomial.
template <int NPOLY, bool PACK>
__global__ void exp2_rate(float* out, long long* clk, int iters) {
  float v[16];
  for (int k = 0; k < 16; ++k) v[k] = 0.5f + 0.01f * k + 1e-4f * threadIdx.x;
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    float x[16];
#pragma unroll
    for (int k = 0; k < 16; k += 2)
      up2(fma2(pk2(v[k], v[k + 1]), pk2(-1.f, -1.f), pk2(-0.25f, -0.25f)), x[k], x[k + 1]);
#pragma unroll
    for (int k = 0; k < 16 - NPOLY; ++k) v[k] = ex2_hw(x[k]);
#pragma unroll
    for (int k = 16 - NPOLY; k < 16; k += 2) exp2_poly2(x[k], x[k + 1], v[k], v[k + 1]);
    if (PACK) {
#pragma unroll
      for (int k = 0; k < 16; k += 2) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[k], v[k + 1]);
        const uint32_t u = *reinterpret_cast<const uint32_t*>(&h);
        v[k] = __uint_as_float((u & 0xffff0000u) | 0x3f000000u);   // keep the chain finite
      }
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float s = 0;
  for (int k = 0; k < 16; ++k) s += v[k];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) clk[blockIdx.x] = t1 - t0;
}

__global__ void exp2_values(const float* x, float* yp, float* yh, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (2 * i + 1 < n) {
    float a, b;
    exp2_poly2(x[2 * i], x[2 * i + 1], a, b);
    yp[2 * i] = a;
    yp[2 * i + 1] = b;
    yh[2 * i] = ex2_hw(x[2 * i]);
    yh[2 * i + 1] = ex2_hw(x[2 * i + 1]);
  }
}

template <int NP, bool PK>
bool run(const char* name, int sms, float* out, long long* clk, int threads) {
  const int iters = 4096;
  for (int rep = 0; rep < 2; ++rep) exp2_rate<NP, PK><<<sms, threads>>>(out, clk, iters);
  const cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    printf("error %s\n", cudaGetErrorString(e));
    return false;
  }
  std::vector<long long> h(sms);
  cudaMemcpy(h.data(), clk, sizeof(long long) * sms, cudaMemcpyDeviceToHost);
  double avg = 0;
  for (long long c : h) avg += c;
  avg /= sms;
  printf("%-32s %3d threads/SM: %6.2f exp2/clk/SM\n", name, threads,
         double(iters) * 16 * threads / avg);
  return true;
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  float* out = nullptr;
  long long* clk = nullptr;
  cudaMalloc(&out, sizeof(float) * sms * 512);
  cudaMalloc(&clk, sizeof(long long) * sms);
  for (int threads : {256, 512}) {
    bool ok = run<0, false>("MUFU only", sms, out, clk, threads) &&
              run<16, false>("polynomial only", sms, out, clk, threads) &&
              run<2, false>("polynomial 2/16", sms, out, clk, threads) &&
              run<4, false>("polynomial 4/16", sms, out, clk, threads) &&
              run<6, false>("polynomial 6/16", sms, out, clk, threads) &&
              run<0, true>("MUFU + bf16 pack", sms, out, clk, threads) &&
              run<2, true>("polynomial 2/16 + bf16 pack", sms, out, clk, threads) &&
              run<4, true>("polynomial 4/16 + bf16 pack", sms, out, clk, threads);
    if (!ok) return 1;
  }
  const int n = 1 << 22;
  std::vector<float> hx(n);
  for (int i = 0; i < n; ++i) hx[i] = -130.f + 131.f * float(i) / float(n - 1);
  float *dx, *dp, *dh;
  cudaMalloc(&dx, sizeof(float) * n);
  cudaMalloc(&dp, sizeof(float) * n);
  cudaMalloc(&dh, sizeof(float) * n);
  cudaMemcpy(dx, hx.data(), sizeof(float) * n, cudaMemcpyHostToDevice);
  exp2_values<<<(n / 2 + 255) / 256, 256>>>(dx, dp, dh, n);
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  std::vector<float> yp(n), yh(n);
  cudaMemcpy(yp.data(), dp, sizeof(float) * n, cudaMemcpyDeviceToHost);
  cudaMemcpy(yh.data(), dh, sizeof(float) * n, cudaMemcpyDeviceToHost);
  double ep = 0, eh = 0, below = 0;
  for (int i = 0; i < n; ++i) {
    const double x = hx[i], ref = exp2(x);
    if (x >= -125.0) {
      ep = fmax(ep, fabs(yp[i] / ref - 1));
      eh = fmax(eh, fabs(yh[i] / ref - 1));
    } else {
      below = fmax(below, double(yp[i]));
    }
  }
  printf("max relative error on [-125, 1]: polynomial %.3e, MUFU %.3e; polynomial below -125: <= %.2e\n",
         ep, eh, below);
  return 0;
}
