// Block quantization of bf16 [B,H,N,d] tensors to e4m3 for the FP8 forward
// ("FlashAttention v1～v4" v3 §3: one scale per computation block instead of
// one per tensor).  A block is 128 consecutive rows of one (batch, head):
//   scale = amax(|x| over the block) / 448 (1 for an all-zero block),
//   code  = e4m3(x * (1 / scale)), round to nearest even, saturating,
// the division, reciprocal and product each rounded to fp32.  V is written
// transposed ([B*H, d, Np], Np = N rounded up to 128, zero codes past N) so
// that the second GEMM of the forward reads it K-major.
//
// Incoherent processing (v3 §3): Q and K may first be multiplied by the same
// random orthogonal matrix, M = diag(s) H / sqrt(d) with H the
// Sylvester-Hadamard matrix and s caller-given signs, so that QM (KM)^T =
// Q K^T while an outlier's energy spreads over all d columns before the
// block scale is taken.  Each row is rotated in fp32: the signs, butterflies
// (a + b, a - b) at strides 1, 2, 4, ..., 64 in that order, then one
// multiplication by fp32(1/sqrt(d)).
#include "fattn_internal.h"
#include "fattn_ptx.cuh"

namespace fattn {

namespace {

constexpr int kQThreads = 256;
constexpr int kD = 128;                  // head dimension of the FP8 path
constexpr int kRowBytes = kD * 2;        // one bf16 row
constexpr int kSlots = 8;                // 16-byte chunks per thread per block
constexpr int kQSmemBytes = 2 * kSlots * kQThreads * 16;   // two blocks in flight

// Which 16-byte chunks of a 128-row block a thread quantizes (slot s < 8):
//   kPlain      rows 8 (tid / 16) + s, chunk tid % 16   (row-major output)
//   kTransposed rows 8 (tid % 16) + s, chunk tid / 16   (column-major output:
//               the 16 lanes of a half warp cover one column's 128 rows)
//   kRotated    row tid / 2, chunk 4 (s / 2) + 2 (tid % 2) + s % 2 (two lanes
//               per row; columns 8 chunk + e have bits e = 0-2, s % 2 = 3,
//               tid % 2 = 4 and s / 2 = 5-6)
// kPlain and kRotated copy their own chunks in; kTransposed copies in the
// kPlain pattern (whole rows per warp) and, after a barrier, reads the
// chunks it quantizes from the other threads' slots.
enum class QMode { kPlain, kTransposed, kRotated };

// Physical 16-byte index of thread t's chunk within a slot plane: an XOR
// swizzle that keeps both the row-major copies and the column-major reads of
// kTransposed free of bank conflicts.
__device__ __forceinline__ int swz(int t) { return t ^ ((t >> 4) & 7); }

template <QMode M>
__device__ __forceinline__ void slot_pos(int tid, int s, int& row, int& chunk) {
  if constexpr (M == QMode::kPlain) {
    row = 8 * (tid >> 4) + s;
    chunk = tid & 15;
  } else if constexpr (M == QMode::kTransposed) {
    row = 8 * (tid & 15) + s;
    chunk = tid >> 4;
  } else {
    row = tid >> 1;
    chunk = 4 * (s >> 1) + 2 * (tid & 1) + (s & 1);
  }
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int Pending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" :: "n"(Pending) : "memory");
}

// Packed pairs of fp32 (f32x2 arithmetic, each lane rounded as the scalar op).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
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
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 p = __bfloat1622float2(h[k]);
    f[2 * k] = p.x;
    f[2 * k + 1] = p.y;
  }
}

// amax over the CTA; every thread gets the result.  ``red`` alternates
// between two arrays from one block to the next so that no thread writes the
// next block's partial maxima before all have read this block's.
__device__ __forceinline__ float block_amax(float amax, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  return amax;
}

__device__ __forceinline__ uint2 encode8(const float* f, float inv) {
  uint2 out;
  out.x = pack_e4m3x4(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                      __fmul_rn(f[3], inv));
  out.y = pack_e4m3x4(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv),
                      __fmul_rn(f[7], inv));
  return out;
}

// Four words holding a 4 x 4 byte block row by row -> the same block column
// by column (byte k of word j = byte j of word k).
__device__ __forceinline__ void transpose4x4_bytes(uint32_t a0, uint32_t a1, uint32_t a2,
                                                   uint32_t a3, uint32_t (&c)[4]) {
  const uint32_t t0 = __byte_perm(a0, a1, 0x5140);   // a0.0 a1.0 a0.1 a1.1
  const uint32_t t1 = __byte_perm(a0, a1, 0x7362);   // a0.2 a1.2 a0.3 a1.3
  const uint32_t t2 = __byte_perm(a2, a3, 0x5140);
  const uint32_t t3 = __byte_perm(a2, a3, 0x7362);
  c[0] = __byte_perm(t0, t2, 0x5410);
  c[1] = __byte_perm(t0, t2, 0x7632);
  c[2] = __byte_perm(t1, t3, 0x5410);
  c[3] = __byte_perm(t1, t3, 0x7632);
}

// Index of the m-th element of f[64] whose bit H is clear.
__host__ __device__ constexpr int lower_index(int m, int H) { return (m / H) * 2 * H + m % H; }

// Butterfly (a + b, a - b) on the pairs of f[64] H apart, two pairs per
// f32x2 operation.
template <int H>
__device__ __forceinline__ void butterfly_in_thread(float (&f)[64]) {
#pragma unroll
  for (int m = 0; m < 32; m += 2) {
    const int l0 = lower_index(m, H), l1 = lower_index(m + 1, H);
    const uint64_t a = pk2(f[l0], f[l1]), b = pk2(f[l0 + H], f[l1 + H]);
    upk2(add2(a, b), f[l0], f[l1]);
    upk2(sub2(a, b), f[l0 + H], f[l1 + H]);
  }
}

struct QBlock {
  int bh, row0, rows;
};

__device__ __forceinline__ QBlock block_at(int blk, int N, int n_tiles) {
  QBlock b;
  b.bh = blk / n_tiles;
  b.row0 = (blk - b.bh * n_tiles) * 128;
  b.rows = min(128, N - b.row0);
  return b;
}

// Persistent over blocks (one block = 128 rows of one head, one scale): each
// thread prefetches its own chunks of the CTA's next block with cp.async
// into a private slot-major shared buffer while it quantizes the current
// one.  Rows past N read as zeros (zero-filled copies), so they give code 0.
template <QMode M>
__global__ void __launch_bounds__(kQThreads, M == QMode::kRotated ? 3 : 2) quantize_kernel(
    const uint8_t* __restrict__ x, const float* __restrict__ signs, uint8_t* __restrict__ codes,
    float* __restrict__ scales, int N, int n_tiles, int n_blocks) {
  extern __shared__ __align__(16) uint4 qbuf[];       // [2][kSlots][kQThreads]
  __shared__ float red[2][kQThreads / 32];
  __shared__ __align__(16) uint32_t smask[kD / 2];     // sign bits per bf16 pair
  const int tid = threadIdx.x;
  constexpr QMode kCopy = M == QMode::kTransposed ? QMode::kPlain : M;

  if constexpr (M == QMode::kRotated) {
    // Multiplying by -1 flips the sign bit, exactly: done on the bf16 words.
    if (tid < kD / 2) {
      const uint32_t lo = __float_as_uint(__ldg(signs + 2 * tid)) >> 31;
      const uint32_t hi = __float_as_uint(__ldg(signs + 2 * tid + 1)) >> 31;
      smask[tid] = (lo << 15) | (hi << 31);
    }
    __syncthreads();
  }

  auto prefetch = [&](int blk, int buf) {
    const QBlock b = block_at(blk, N, n_tiles);
    const uint8_t* xb = x + (static_cast<size_t>(b.bh) * N + b.row0) * kRowBytes;
    const int ps = M == QMode::kTransposed ? swz(tid) : tid;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
      int r, c;
      slot_pos<kCopy>(tid, s, r, c);
      const bool in = r < b.rows;
      cp_async16(&qbuf[(buf * kSlots + s) * kQThreads + ps], in ? xb + r * kRowBytes + c * 16 : xb,
                 in ? 16 : 0);
    }
    cp_async_commit();
  };

  int blk = blockIdx.x;
  if (blk < n_blocks) prefetch(blk, 0);
  for (int it = 0; blk < n_blocks; ++it, blk += gridDim.x) {
    const int nxt = blk + gridDim.x;
    if (nxt < n_blocks) {
      prefetch(nxt, (it + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    uint4 raw[kSlots];
    if constexpr (M == QMode::kTransposed) {
      __syncthreads();                      // every thread's copies of this block landed
      const int src = swz(16 * (tid & 15) + (tid >> 4));
#pragma unroll
      for (int s = 0; s < kSlots; ++s) raw[s] = qbuf[((it & 1) * kSlots + s) * kQThreads + src];
    } else {
#pragma unroll
      for (int s = 0; s < kSlots; ++s) raw[s] = qbuf[((it & 1) * kSlots + s) * kQThreads + tid];
    }
    const QBlock b = block_at(blk, N, n_tiles);

    if constexpr (M == QMode::kRotated) {
      float f[64];
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        int r, c;
        slot_pos<M>(tid, s, r, c);
        const uint4 m = reinterpret_cast<const uint4*>(smask)[c];
        uint4 v = raw[s];
        v.x ^= m.x;
        v.y ^= m.y;
        v.z ^= m.z;
        v.w ^= m.w;
        bf16x8_to_f32(v, &f[8 * s]);
      }
#pragma unroll
      for (int j = 0; j < 64; j += 2) {    // column stride 1: a pair's own halves
        const float a = f[j], b = f[j + 1];
        f[j] = __fadd_rn(a, b);
        f[j + 1] = __fsub_rn(a, b);
      }
      butterfly_in_thread<2>(f);           // column strides 2, 4, 8
      butterfly_in_thread<4>(f);
      butterfly_in_thread<8>(f);
      {                                     // column stride 16: the other lane
        const float c = (tid & 1) ? -1.f : 1.f;   // upper lane: other - mine
        const uint64_t cc = pk2(c, c);
#pragma unroll
        for (int m = 0; m < 64; m += 2) {
          const float o0 = __shfl_xor_sync(0xffffffffu, f[m], 1);
          const float o1 = __shfl_xor_sync(0xffffffffu, f[m + 1], 1);
          upk2(fma2(pk2(f[m], f[m + 1]), cc, pk2(o0, o1)), f[m], f[m + 1]);
        }
      }
      butterfly_in_thread<16>(f);          // column strides 32, 64
      butterfly_in_thread<32>(f);
      constexpr float kInvSqrt128 = 0.08838834764831845f;
      const uint64_t k2 = pk2(kInvSqrt128, kInvSqrt128);
      float amax = 0.f;
#pragma unroll
      for (int m = 0; m < 64; m += 2) {
        upk2(mul2(pk2(f[m], f[m + 1]), k2), f[m], f[m + 1]);
        amax = fmaxf(amax, fmaxf(fabsf(f[m]), fabsf(f[m + 1])));
      }
      amax = block_amax(amax, red[it & 1]);
      const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      const float inv = __fdiv_rn(1.f, sc);
      if (tid == 0) scales[blk] = sc;
      const int r = tid >> 1;
      if (r < b.rows) {
        uint8_t* dst = codes + (static_cast<size_t>(b.bh) * N + b.row0 + r) * kD;
        const uint64_t inv2 = pk2(inv, inv);
#pragma unroll
        for (int m = 0; m < 64; m += 2) upk2(mul2(pk2(f[m], f[m + 1]), inv2), f[m], f[m + 1]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {      // slots 2j, 2j + 1: 16 adjacent codes
          const uint4 w = make_uint4(pack_e4m3x4(f[16 * j], f[16 * j + 1], f[16 * j + 2], f[16 * j + 3]),
                                     pack_e4m3x4(f[16 * j + 4], f[16 * j + 5], f[16 * j + 6], f[16 * j + 7]),
                                     pack_e4m3x4(f[16 * j + 8], f[16 * j + 9], f[16 * j + 10], f[16 * j + 11]),
                                     pack_e4m3x4(f[16 * j + 12], f[16 * j + 13], f[16 * j + 14], f[16 * j + 15]));
          *reinterpret_cast<uint4*>(dst + (4 * j + 2 * (tid & 1)) * 8) = w;
        }
      }
    } else {
      float amax = 0.f;
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        float f[8];
        bf16x8_to_f32(raw[s], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
      }
      amax = block_amax(amax, red[it & 1]);
      const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      const float inv = __fdiv_rn(1.f, sc);
      if (tid == 0) scales[blk] = sc;
      uint2 q[kSlots];
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        float f[8];
        bf16x8_to_f32(raw[s], f);
        q[s] = encode8(f, inv);
      }
      if constexpr (M == QMode::kPlain) {
        const int r8 = 8 * (tid >> 4), c8 = tid & 15;
#pragma unroll
        for (int s = 0; s < kSlots; ++s)
          if (r8 + s < b.rows)
            *reinterpret_cast<uint2*>(
                codes + (static_cast<size_t>(b.bh) * N + b.row0 + r8 + s) * kD + c8 * 8) = q[s];
      } else {
        const int r8 = 8 * (tid & 15), c8 = tid >> 4;
        uint32_t lo[2][4], hi[2][4];        // [row quad][column within the half]
#pragma unroll
        for (int rq = 0; rq < 2; ++rq) {
          transpose4x4_bytes(q[4 * rq].x, q[4 * rq + 1].x, q[4 * rq + 2].x, q[4 * rq + 3].x,
                             lo[rq]);
          transpose4x4_bytes(q[4 * rq].y, q[4 * rq + 1].y, q[4 * rq + 2].y, q[4 * rq + 3].y,
                             hi[rq]);
        }
        const size_t np = static_cast<size_t>(n_tiles) * 128;
        uint8_t* col0 = codes + (static_cast<size_t>(b.bh) * kD + c8 * 8) * np + b.row0 + r8;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          *reinterpret_cast<uint2*>(col0 + j * np) = make_uint2(lo[0][j], lo[1][j]);
          *reinterpret_cast<uint2*>(col0 + (j + 4) * np) = make_uint2(hi[0][j], hi[1][j]);
        }
      }
    }
  }
}

template <QMode M>
cudaError_t launch_quantize(const void* x, const float* signs, void* codes, float* scales,
                            int BH, int N, cudaStream_t stream) {
  auto kern = quantize_kernel<M>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int n_tiles = (N + 127) / 128;
  const long long blocks = static_cast<long long>(BH) * n_tiles;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  // Two CTAs per SM (three for the rotation: latency-bound, it gains from
  // the extra warps), each looping over blocks.
  const long long per_sm = M == QMode::kRotated ? 3 : 2;
  const long long grid = blocks < per_sm * sms ? blocks : per_sm * sms;
  kern<<<static_cast<unsigned>(grid), kQThreads, kQSmemBytes, stream>>>(
      static_cast<const uint8_t*>(x), signs, static_cast<uint8_t*>(codes), scales, N, n_tiles,
      static_cast<int>(blocks));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_quantize_rotated(const void* x, const float* signs, void* codes,
                                        float* scales, int BH, int N, int d,
                                        cudaStream_t stream) {
  if (d != kD || signs == nullptr) return cudaErrorInvalidValue;
  return launch_quantize<QMode::kRotated>(x, signs, codes, scales, BH, N, stream);
}

cudaError_t launch_fp8_quantize(const void* x, void* codes, float* scales, int BH, int N, int d,
                                bool transpose, cudaStream_t stream) {
  if (d != kD) return cudaErrorInvalidValue;
  return transpose
             ? launch_quantize<QMode::kTransposed>(x, nullptr, codes, scales, BH, N, stream)
             : launch_quantize<QMode::kPlain>(x, nullptr, codes, scales, BH, N, stream);
}

}  // namespace fattn
