// Microbenchmark: per-SM throughput of global -> shared loads from an
// L2-resident 8 MiB buffer, the traffic that feeds the K/V ring of the forward
// and the Q/dO ring of the backward.  One CTA per SM.
//   tma      cp.async.bulk.tensor of 128-byte-swizzled boxes (128-byte rows),
//            each issuing warp keeping 4 boxes in flight in its own ring of
//            shared-memory slots; box height and warp count vary the bytes in
//            flight
//   cp.async 16 bytes per thread (.cg), 16 KiB per group, 4 groups in flight,
//            from a growing number of warps
// Every mbarrier wait is bounded; a CTA that gives up reports 0 cycles and is
// counted as a timeout.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <vector>

namespace {

constexpr size_t kBufBytes = 8u << 20;
constexpr int kSlots = 4;
constexpr long long kSpinLimit = 1ll << 26;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool wait_parity(uint32_t bar, uint32_t parity) {
  for (long long spins = 0; spins < kSpinLimit; ++spins) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity));
    if (done) return true;
  }
  return false;
}

// Lane 0 of each warp streams `iters` boxes of box_rows x 128 bytes.
__global__ void tma_rate(const __grid_constant__ CUtensorMap tm, int iters, int nbox, int box_rows,
                         unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* buf = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t bars[2 * kSlots];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int box_bytes = box_rows * 128;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * kSlots; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[i])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const unsigned long long t0 = clock64();
  bool ok = true;
  if (lane == 0) {
    int issued = 0;
    for (int it = 0; ok && it < iters + kSlots; ++it) {
      const int s = kSlots * warp + (it % kSlots);
      const uint32_t bar = smem_addr(&bars[s]);
      if (it >= kSlots) ok = wait_parity(bar, ((it - kSlots) / kSlots) & 1);
      if (ok && it < iters) {
        ++issued;
        const int box = (blockIdx.x * 7 + it * 3 + warp * 101) % nbox;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"(box_bytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(buf + s * box_bytes)),
            "l"(reinterpret_cast<uint64_t>(&tm)), "r"(0), "r"(box * box_rows), "r"(bar)
            : "memory");
      }
    }
    // After a timeout, let this warp's last copies land (bounded) before exit.
    if (!ok)
      for (int it = issued > kSlots ? issued - kSlots : 0; it < issued; ++it)
        wait_parity(smem_addr(&bars[kSlots * warp + (it % kSlots)]), (it / kSlots) & 1);
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  __shared__ int any_fail;
  if (threadIdx.x == 0) any_fail = 0;
  __syncthreads();
  if (!ok) atomicOr(&any_fail, 1);
  __syncthreads();
  if (threadIdx.x == 0) cycles[blockIdx.x] = any_fail ? 0ull : t1 - t0;
}

// Every thread copies 16-byte pieces of one 16 KiB block per group.
__global__ void cp_async_rate(const uint8_t* __restrict__ src, int iters,
                              unsigned long long* cycles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* buf = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int nblk = static_cast<int>(kBufBytes / 16384);
  __syncthreads();
  const unsigned long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
    const uint8_t* s = src + static_cast<size_t>((blockIdx.x * 13 + it * 3) % nblk) * 16384;
    uint8_t* d = buf + (it % kSlots) * 16384;
    for (int c = threadIdx.x; c < 1024; c += blockDim.x)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(d + c * 16)),
                   "l"(s + c * 16)
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 3;" ::: "memory");
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();
  const unsigned long long t1 = clock64();
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

bool check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) std::printf("%s: %s\n", what, cudaGetErrorString(e));
  return e == cudaSuccess;
}

}  // namespace

int main() {
  uint8_t* src = nullptr;
  if (!check(cudaMalloc(&src, kBufBytes), "cudaMalloc")) return 1;
  if (!check(cudaMemset(src, 1, kBufBytes), "cudaMemset")) return 1;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* dcyc = nullptr;
  if (!check(cudaMalloc(&dcyc, sizeof(unsigned long long) * sms), "cudaMalloc")) return 1;
  std::vector<unsigned long long> cyc(sms);
  const int iters = 2048;
  const int rows_total = static_cast<int>(kBufBytes / 128);

  struct TmaCase { int rows, warps; };
  for (const TmaCase c : {TmaCase{64, 1}, TmaCase{128, 1}, TmaCase{64, 2}, TmaCase{256, 1},
                          TmaCase{128, 2}}) {
    CUtensorMap tm;
    cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows_total)};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(c.rows)};
    cuuint32_t es[2] = {1, 1};
    if (cuTensorMapEncodeTiled(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, src, dims, strides, box, es,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      std::printf("cuTensorMapEncodeTiled failed\n");
      return 1;
    }
    const int box_bytes = c.rows * 128;
    const int smem = c.warps * kSlots * box_bytes + 1024;
    if (!check(cudaFuncSetAttribute(tma_rate, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
               "smem attribute"))
      return 1;
    for (int rep = 0; rep < 2; ++rep)
      tma_rate<<<sms, 32 * c.warps, smem>>>(tm, iters, rows_total / c.rows, c.rows, dcyc);
    if (!check(cudaGetLastError(), "launch") || !check(cudaDeviceSynchronize(), "tma_rate"))
      return 1;
    cudaMemcpy(cyc.data(), dcyc, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost);
    double sum = 0;
    int timeouts = 0;
    for (int b = 0; b < sms; ++b) {
      sum += static_cast<double>(cyc[b]);
      timeouts += cyc[b] == 0;
    }
    const double in_flight = static_cast<double>(c.warps) * kSlots * box_bytes;
    const double rate = static_cast<double>(iters) * c.warps * box_bytes / (sum / sms);
    std::printf("tma      box %3d rows x 128 B, %d warp(s): %5.1f KiB in flight  %5.1f B/clk/SM"
                "  (in flight / rate = %4.0f clk)%s\n",
                c.rows, c.warps, in_flight / 1024, rate, in_flight / rate,
                timeouts ? "  TIMEOUTS" : "");
  }
  for (const int warps : {2, 4, 8, 16}) {
    const int smem = kSlots * 16384 + 1024;
    if (!check(cudaFuncSetAttribute(cp_async_rate, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem),
               "smem attribute"))
      return 1;
    for (int rep = 0; rep < 2; ++rep) cp_async_rate<<<sms, 32 * warps, smem>>>(src, iters, dcyc);
    if (!check(cudaGetLastError(), "launch") || !check(cudaDeviceSynchronize(), "cp_async_rate"))
      return 1;
    cudaMemcpy(cyc.data(), dcyc, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost);
    double sum = 0;
    for (int b = 0; b < sms; ++b) sum += static_cast<double>(cyc[b]);
    std::printf("cp.async 16 B per thread, %2d warps, 4 x 16 KiB groups in flight: %5.1f B/clk/SM\n",
                warps, static_cast<double>(iters) * 16384 / (sum / sms));
  }
  return 0;
}
