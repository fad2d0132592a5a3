// Microbenchmark: per-SM throughput of fp32 reduce-adds into global memory,
// the operation that accumulates dQ across K/V tiles.  Every CTA adds into a
// private 64 KiB region (no two SMs touch the same line), with
//   red.f32      one 4-byte add per lane, 128 bytes per warp instruction
//   red.v4.f32   16 bytes per lane, 512 contiguous bytes per instruction
//   bulk         cp.reduce.async.bulk .add.f32 from shared memory, 4 KiB per
//                copy, at most four copies in flight (the async-proxy path)
// for a growing number of SMs.
#include <cstdint>
#include <cstdio>
#include <vector>
#include <cuda_runtime.h>

namespace {

constexpr int kRegionFloats = 16384;   // 64 KiB per CTA

__global__ void reduce_rate(float* buf, long long* out, int iters, int mode) {
  extern __shared__ __align__(128) float src[];   // 4 KiB of ones (bulk mode)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* base = buf + static_cast<size_t>(blockIdx.x) * kRegionFloats;
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) src[i] = 1.0f;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  const long long t0 = clock64();
  if (mode == 0) {
    for (int i = 0; i < iters; ++i) {
      float* p = base + (((i * 8 + warp) * 32) % kRegionFloats) + lane;
      asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(1.0f) : "memory");
    }
  } else if (mode == 1) {
    for (int i = 0; i < iters; ++i) {
      float* p = base + (((i * 8 + warp) * 128) % kRegionFloats) + lane * 4;
      asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %1, %1, %1};" ::"l"(p), "f"(1.0f)
                   : "memory");
    }
  } else if (threadIdx.x == 0) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(src));
    for (int i = 0; i < iters; ++i) {
      float* p = base + ((i * 1024) % kRegionFloats);
      asm volatile(
          "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], 4096;" ::"l"(p),
          "r"(s)
          : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  __syncthreads();
  const long long t1 = clock64();
  if (threadIdx.x == 0) out[blockIdx.x] = t1 - t0;
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int threads = 256;
  const size_t bytes = static_cast<size_t>(sms) * kRegionFloats * sizeof(float);
  float* buf = nullptr;
  cudaMalloc(&buf, bytes);
  cudaMemset(buf, 0, bytes);
  long long* out = nullptr;
  cudaMalloc(&out, sizeof(long long) * sms);
  std::vector<long long> h(sms);
  const char* names[3] = {"red.f32     (128 B/instr)", "red.v4.f32  (512 B/instr)",
                          "bulk reduce (4 KiB/copy) "};
  for (int mode = 0; mode < 3; ++mode) {
    // bytes added per CTA: warps x iters x bytes per instruction, or iters x 4 KiB
    const int iters = mode == 2 ? 4096 : 4096;
    const double per_cta = mode == 0   ? double(iters) * (threads / 32) * 128
                           : mode == 1 ? double(iters) * (threads / 32) * 512
                                       : double(iters) * 4096;
    for (int g : {1, 8, 38, 76, sms}) {
      for (int rep = 0; rep < 2; ++rep) reduce_rate<<<g, threads, 4096>>>(buf, out, iters, mode);
      const cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) {
        printf("error %s\n", cudaGetErrorString(e));
        return 1;
      }
      cudaMemcpy(h.data(), out, sizeof(long long) * g, cudaMemcpyDeviceToHost);
      double avg = 0;
      for (int b = 0; b < g; ++b) avg += h[b];
      avg /= g;
      printf("%s  SMs %3d: %5.1f B/clk/SM\n", names[mode], g, per_cta / avg);
    }
  }
  return 0;
}
