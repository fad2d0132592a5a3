// Microbenchmark: cost of one tcgen05.mma (bf16 in, fp32 accumulate in TMEM)
// for the shapes the attention kernels use, one CTA per SM, issued back to
// back.  Operand contents do not affect the timing (the shared-memory tiles
// are left uninitialised).
//
// Cases: SS (both operands in shared memory) and TS (A from TMEM) at
// 128x128x16, SS at 128x256x16; issued by the kernels' converged-warp form
// (the whole warp runs it, elect.sync picks the issuing lane) or by lane 0
// alone; with 1, 2 or 4 accumulators in TMEM used in turn -- with one, every
// MMA accumulates onto the previous one's result, as the K steps of one GEMM
// do; with several, consecutive MMAs are independent, as the K steps of
// interleaved GEMMs would be; alone, or with 8 warps of FMAs competing for
// issue slots.  Everything is unrolled at compile time and the descriptors are
// built once, as in the kernels.
#include <cstdint>
#include <cstdio>
#include <vector>
#include <cuda_runtime.h>

#include "../csrc/fattn_ptx.cuh"
using namespace fattn;

namespace {

// Single-thread issue forms (the kernels use the converged-warp `_w` forms of
// fattn_ptx.cuh; these time the other way of issuing).
// D(tmem) (+)= A(smem) * B(smem)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 MMA issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

enum Kind { kSS128 = 0, kTS128 = 1, kSS256 = 2 };

template <int KIND, int NACC, bool CONVERGED, bool BUSY>
__global__ void __launch_bounds__(384, 1) mma_rate(long long* out, int iters) {
  static_assert(NACC * (KIND == kSS256 ? 256 : 128) <= (KIND == kTS128 ? 256 : 512),
                "accumulators must fit in TMEM (TS keeps its A operand at columns 256+)");
  constexpr int kN = KIND == kSS256 ? 256 : 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tbase;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sA = (smem_u32(smem) + 1023u) & ~1023u, sB = sA + 32768;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tbase), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tbase;
  if (warp == 0 && (CONVERGED || lane == 0)) {
    constexpr bool kTs = KIND == kTS128;
    constexpr uint32_t idesc = idesc_bf16_f32(128, kN, false, kTs);
    const uint64_t da = sdesc_sw128(sA, 16, 1024);
    const uint64_t db = kTs ? sdesc_sw128(sB, 16384, 1024) : sdesc_sw128(sB, 16, 1024);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        constexpr uint32_t kChunkB = kN == 256 ? 32768 : 16384;
        const uint32_t offa = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
        const uint32_t offb = kTs ? ((kk * 2048) >> 4) : ((kk >> 2) * kChunkB + (kk & 3) * 32) >> 4;
#pragma unroll
        for (int a = 0; a < NACC; ++a) {
          const uint32_t d = tmem + static_cast<uint32_t>(a * kN);
          if (kTs) {
            if (CONVERGED)
              mma_ts_w(d, tmem + 256 + 8 * kk, db + offb, idesc, 1u);
            else
              mma_ts(d, tmem + 256 + 8 * kk, db + offb, idesc, 1u);
          } else {
            if (CONVERGED)
              mma_ss_w(d, da + offa, db + offb, idesc, 1u);
            else
              mma_ss(d, da + offa, db + offb, idesc, 1u);
          }
        }
      }
    }
    const long long t1 = clock64();
    if (CONVERGED) {
      mma_commit_w(smem_u32(&bar));
    } else {
      mma_commit(smem_u32(&bar));
    }
    long long spins = 0;   // bounded: the MMAs above complete in well under a millisecond
    while (!mbar_try_wait(smem_u32(&bar), 0) && spins < (1ll << 26)) ++spins;
    const long long t2 = clock64();
    if (lane == 0) {
      out[blockIdx.x * 4 + 0] = t1 - t0;
      out[blockIdx.x * 4 + 1] = t2 - t0;
      out[blockIdx.x * 4 + 2] = spins;
    }
  } else if (BUSY && warp >= 1 && warp <= 8) {
    float a0 = lane, a1 = lane + 1, a2 = lane + 2, a3 = lane + 3;
    for (int i = 0; i < iters * NACC * 64; ++i) {
      a0 = fmaf(a0, 1.0001f, 0.5f);
      a1 = fmaf(a1, 1.0001f, 0.5f);
      a2 = fmaf(a2, 1.0001f, 0.5f);
      a3 = fmaf(a3, 1.0001f, 0.5f);
    }
    if (a0 + a1 + a2 + a3 == 1.2345f) out[blockIdx.x * 4 + 3] = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

struct Case {
  const char* name;
  void (*kernel)(long long*, int);
  int n, n_acc;
};

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  long long* d = nullptr;
  cudaMalloc(&d, sizeof(long long) * 4 * sms);
  cudaMemset(d, 0, sizeof(long long) * 4 * sms);
  const int smem = 32768 + 65536 + 1024;
  const Case cases[] = {
      {"SS 128x128x16, converged, 1 acc", mma_rate<kSS128, 1, true, false>, 128, 1},
      {"SS 128x128x16, converged, 2 acc", mma_rate<kSS128, 2, true, false>, 128, 2},
      {"SS 128x128x16, converged, 4 acc", mma_rate<kSS128, 4, true, false>, 128, 4},
      {"SS 128x128x16, lane 0, 1 acc", mma_rate<kSS128, 1, false, false>, 128, 1},
      {"SS 128x128x16, lane 0, 2 acc", mma_rate<kSS128, 2, false, false>, 128, 2},
      {"TS 128x128x16, converged, 1 acc", mma_rate<kTS128, 1, true, false>, 128, 1},
      {"TS 128x128x16, converged, 2 acc", mma_rate<kTS128, 2, true, false>, 128, 2},
      {"SS 128x256x16, converged, 1 acc", mma_rate<kSS256, 1, true, false>, 256, 1},
      {"SS 128x256x16, converged, 2 acc", mma_rate<kSS256, 2, true, false>, 256, 2},
      {"SS 128x128x16, converged, 1 acc, 8 FMA warps", mma_rate<kSS128, 1, true, true>, 128, 1},
      {"SS 128x128x16, converged, 2 acc, 8 FMA warps", mma_rate<kSS128, 2, true, true>, 128, 2},
  };
  const int mmas = 2048;   // per CTA and case
  std::vector<long long> h(4 * sms);
  for (const Case& cs : cases) {
    cudaFuncSetAttribute(cs.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const int iters = mmas / (8 * cs.n_acc);
    for (int rep = 0; rep < 2; ++rep) {
      cs.kernel<<<sms, 384, smem>>>(d, iters);
      const cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) {
        printf("error %s\n", cudaGetErrorString(e));
        return 1;
      }
    }
    cudaMemcpy(h.data(), d, sizeof(long long) * 4 * sms, cudaMemcpyDeviceToHost);
    double issue = 0, total = 0;
    long long spins = 0;
    for (int b = 0; b < sms; ++b) {
      issue += h[4 * b];
      total += h[4 * b + 1];
      spins = spins > h[4 * b + 2] ? spins : h[4 * b + 2];
    }
    issue /= sms;
    total /= sms;
    const int n = iters * 8 * cs.n_acc;
    const double flop = 2.0 * 128 * cs.n * 16;
    printf("%-46s issue %6.1f clk/MMA  complete %6.1f clk/MMA  -> %5.0f FLOP/clk/SM%s\n", cs.name,
           issue / n, total / n, flop * n / total, spins >= (1ll << 26) ? "  (wait limit hit)" : "");
  }
  return 0;
}
