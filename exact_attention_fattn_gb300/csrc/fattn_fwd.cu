// Forward pass of exact attention on sm_103a: TMA producer -> shared-memory
// K/V ring -> single-thread tcgen05 MMA issuer -> softmax warpgroups over
// TMEM.
//
// Algorithm ("6.1 FlashAttention V1详解" §3.2 online softmax; "FlashAttention
// v1～v4" v1 §2 pseudocode with Q blocks outer, v2 §1 deferred normalisation
// and L = m + log l, v4 §1 accumulators in tensor memory, v4 §3 conditional
// rescaling): for each 128-row Q tile, walk the 128-row K/V tiles j, with
//   S = Q K_j^T                               (tcgen05, fp32 in TMEM)
//   m_new = max(m, rowmax S)                  (softmax thread, one per row)
//   P = 2^(S*scale*log2e - m_ref)             (bf16 back into TMEM)
//   l = alpha*l + rowsum P,  O = alpha*O + P V_j  (tcgen05, O in TMEM)
// and O/l, L are written once at the end.
//
// CTA = two Q tiles (rows [256*pair, 256*pair + 256)) of one (batch, head):
//   warps 0-3  softmax for Q tile 0 (TMEM lanes 0..127, one row per thread)
//   warps 4-7  softmax for Q tile 1
//   warp 8     TMEM allocation + MMA issue (lane 0)
//   warp 9     TMA producer (lane 0)
//   warps 10-11 idle
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+d) O1 [256+d,256+2d);
// P_t (bf16 pairs, 64 columns) aliases S_t at d = 128 and sits in
// [384+64t, 448+64t) at d = 64.
#include "fattn_internal.h"
#include "fattn_ptx.cuh"

namespace fattn {

namespace {

constexpr int kBM = 128;            // rows per Q tile
constexpr int kBN = 128;            // rows per K/V tile
constexpr int kThreads = 384;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr float kLn2 = 0.69314718055994530942f;
// Register split: the kernel launches with kLaunchRegs per thread (384 x 168 =
// 64,512); the control warpgroup (warps 8-11) gives back down to kCtrlRegs and
// the two softmax warpgroups grow to kSoftmaxRegs: 128 x 72 + 256 x 216 =
// 64,512, exactly the launch total, so setmaxnreg.inc can always complete.
constexpr int kLaunchRegs = 168;
constexpr int kCtrlRegs = 72;
constexpr int kSoftmaxRegs = 216;
static_assert(128 * kCtrlRegs + 256 * kSoftmaxRegs == kThreads * kLaunchRegs, "register split");

template <int HD>
struct FwdCfg {
  static constexpr int kChunks = HD / 64;               // 128-byte swizzle chunks per row
  static constexpr int kChunkBytes = kBM * 128;         // one chunk of a 128-row tile
  static constexpr int kTileBytes = kBM * HD * 2;
  static constexpr int kStages = HD == 128 ? 4 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kKvOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKvOff + kStages * kTileBytes;
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + HD * t; }
  __device__ static constexpr uint32_t col_p(int t) {
    return HD == 128 ? 128u * t : 384u + 64u * t;
  }
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct FwdBars {
  uint32_t q_full, kv_full0, kv_empty0, s_full[2], p_full[2], o_full[2], mma_done;
};

template <int HD, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdArgs args) {
  using C = FwdCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kBarOff;
  FwdBars b;
  b.q_full = bar0;
  b.kv_full0 = bar0 + 8;
  b.kv_empty0 = bar0 + 8 * (1 + C::kStages);
  const uint32_t rest = bar0 + 8 * (1 + 2 * C::kStages);
  b.s_full[0] = rest;
  b.s_full[1] = rest + 8;
  b.p_full[0] = rest + 16;
  b.p_full[1] = rest + 24;
  b.o_full[0] = rest + 32;
  b.o_full[1] = rest + 40;
  b.mma_done = rest + 48;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work of this CTA: a pair of Q tiles of one (batch, head).  The
  // pairs with the most key tiles (causal) are launched first.
  const int N = args.N;
  const int num_pairs = (N + 2 * kBM - 1) / (2 * kBM);
  const int bh = blockIdx.x % args.BH;
  const int pair = num_pairs - 1 - static_cast<int>(blockIdx.x / args.BH);
  const int q0 = pair * 2 * kBM;
  const int n_kv = (N + kBN - 1) / kBN;
  int n_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qs = q0 + t * kBM;
    n_t[t] = qs >= N ? 0 : (CAUSAL ? min(n_kv, qs / kBN + 1) : n_kv);
  }
  const int nt = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    mbar_init(b.q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(b.kv_full0 + 8 * s, 1);
      mbar_init(b.kv_empty0 + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(b.s_full[t], 1);
      mbar_init(b.p_full[t], 4 * 32);
      mbar_init(b.o_full[t], 1);
    }
    mbar_init(b.mma_done, 1);
    misc[1] = 0u;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&misc[0]), 512);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtx wc{args.wait_budget, reinterpret_cast<volatile uint32_t*>(&misc[1]), args.status};

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ================================================================ softmax
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r_tile = wq * 32 + lane;
    const int qs = q0 + t * kBM;
    const int row = qs + r_tile;
    const int nj = n_t[t];
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(t);
    const uint32_t tP = tmem + lane_off + C::col_p(t);
    const uint32_t tO = tmem + lane_off + C::col_o(t);
    const float c = args.scale_log2;
    const float tau = args.tau_log2;
    float m_ref = -INFINITY;  // running reference max, log2 units
    float l = 0.f;            // sum of the fp32 probabilities (gives L)
    float l_bf = 0.f;         // sum of their bf16 roundings (normalises O)
    bool ok = true;
    for (int j = 0; j < nj; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(b.s_full[t], j & 1, wc, kWaitSFull));
      if (!ok) break;
      tc_fence_after();
      uint32_t s0[32], s1[32], s2[32], s3[32];
      tmem_ld32(tS + 0, s0);
      tmem_ld32(tS + 32, s1);
      tmem_ld32(tS + 64, s2);
      tmem_ld32(tS + 96, s3);
      tmem_ld_wait32(s0);
      reg_fence32(s1);
      reg_fence32(s2);
      reg_fence32(s3);
      uint32_t* sv[4] = {s0, s1, s2, s3};
      const int kv0 = j * kBN;
      const bool need_mask = (kv0 + kBN > N) || (CAUSAL && kv0 + kBN - 1 > qs);
      if (need_mask) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int col = kv0 + g * 32 + i;
            if (col >= N || (CAUSAL && col > row)) sv[g][i] = __float_as_uint(-INFINITY);
          }
        }
      }
      // Row max as four independent 3-input max chains (one per 32-column
      // group), so the reduction is not one 128-long dependent chain.
      float mg[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float a = fmax3(__uint_as_float(sv[g][0]), __uint_as_float(sv[g][1]),
                        __uint_as_float(sv[g][2]));
        float b2 = fmax3(__uint_as_float(sv[g][3]), __uint_as_float(sv[g][4]),
                         __uint_as_float(sv[g][5]));
#pragma unroll
        for (int i = 6; i < 30; i += 4) {
          a = fmax3(a, __uint_as_float(sv[g][i]), __uint_as_float(sv[g][i + 1]));
          b2 = fmax3(b2, __uint_as_float(sv[g][i + 2]), __uint_as_float(sv[g][i + 3]));
        }
        mg[g] = fmax3(a, b2, fmaxf(__uint_as_float(sv[g][30]), __uint_as_float(sv[g][31])));
      }
      const float mx = fmaxf(fmax3(mg[0], mg[1], mg[2]), mg[3]);
      const float m_new = mx * c;
      const bool need = m_new > m_ref + tau;
      if (__any_sync(0xffffffffu, need)) {
        // O must be rescaled by alpha = 2^(m_old - m_new) before P V_j is
        // added.  P V_{j-1} has completed: it was issued before S_j, whose
        // completion we just waited for.
        const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
        if (need) m_ref = m_new;
        l *= alpha;
        l_bf *= alpha;
        if (j > 0) {
#pragma unroll 1
          for (int ch = 0; ch < HD / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * ch, o);
            tmem_ld_wait32(o);
            const uint64_t a2 = splat2(alpha);
#pragma unroll
            for (int i = 0; i < 16; ++i) unpack2(fmul2(pack2(o[2 * i], o[2 * i + 1]), a2), o[2 * i], o[2 * i + 1]);
            tmem_st32(tO + 32 * ch, o);
          }
        }
      }
      const uint64_t c2 = splat2(c);
      const uint64_t nm2 = splat2(-m_ref);
      // Two columns per instruction (packed fp32 pairs); partial sums per
      // 32-column group keep the additions independent.
      uint64_t rs2[4], rb2[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t pk[16];
        uint64_t e2 = 0ull, b2 = 0ull;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t x0, x1;
          unpack2(ffma2(pack2(sv[g][2 * i], sv[g][2 * i + 1]), c2, nm2), x0, x1);
          const float a0 = ex2_approx(__uint_as_float(x0));
          const float a1 = ex2_approx(__uint_as_float(x1));
          pk[i] = pack_bf16x2(a0, a1);
          e2 = fadd2(e2, pack2(__float_as_uint(a0), __float_as_uint(a1)));
          // O is divided by the sum of the bf16 values that P V actually
          // used, so that O is a convex combination of V rows with the
          // rounded weights (exact for a row dominated by one key); L keeps
          // the fp32 sum.
          b2 = fadd2(b2, pack2(pk[i] << 16, pk[i] & 0xffff0000u));
        }
        tmem_st16(tP + 16 * g, pk);
        rs2[g] = e2;
        rb2[g] = b2;
      }
      float rs[4], rs_bf[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t u0, u1;
        unpack2(rs2[g], u0, u1);
        rs[g] = __uint_as_float(u0) + __uint_as_float(u1);
        unpack2(rb2[g], u0, u1);
        rs_bf[g] = __uint_as_float(u0) + __uint_as_float(u1);
      }
      l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      l_bf += (rs_bf[0] + rs_bf[1]) + (rs_bf[2] + rs_bf[3]);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b.p_full[t]);
    }
    if (ok && nj > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(b.o_full[t], 0, wc, kWaitOFull));
      if (ok) {
        tc_fence_after();
        if (row < N) args.lse[static_cast<size_t>(bh) * N + row] = (m_ref + log2f(l)) * kLn2;
        const float inv = 1.f / l_bf;
        // Stage the bf16 tile in Q_t's shared memory (all MMAs reading Q_t
        // have completed) with the 128-byte swizzle the TMA store expects.
        const uint32_t stage = sbase + C::kQOff + t * C::kTileBytes;
#pragma unroll 1
        for (int ch = 0; ch < HD / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * ch, o);
          tmem_ld_wait32(o);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
          const uint32_t rowaddr = stage + (ch >> 1) * C::kChunkBytes + r_tile * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t chunk = (ch & 1) * 4 + q;
            st_shared_v4(rowaddr + ((chunk ^ (r_tile & 7)) << 4), pk[4 * q], pk[4 * q + 1],
                         pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && qs + wq * 32 < N) {
#pragma unroll
          for (int cc = 0; cc < C::kChunks; ++cc)
            tma_store_3d(&tm_o, stage + cc * C::kChunkBytes + wq * 32 * 128, cc * 64,
                         qs + wq * 32, bh);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        __syncwarp();
      }
    }
  } else if (warp == kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ MMA issue
    // The whole warp runs this (converged); one elected lane issues.
    {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, HD, false, true);
      auto kv_smem = [&](int i) {
        return sbase + C::kKvOff + static_cast<uint32_t>(i % C::kStages) * C::kTileBytes;
      };
      auto kv_full = [&](int i) { return b.kv_full0 + 8u * (i % C::kStages); };
      auto kv_empty = [&](int i) { return b.kv_empty0 + 8u * (i % C::kStages); };
      auto kv_parity = [&](int i) { return static_cast<uint32_t>((i / C::kStages) & 1); };
      // S_t = Q_t K^T: M = 128, N = 128, K = HD in steps of 16 (32 bytes
      // inside a 128-byte swizzle row, then the next 64-column chunk).  The
      // descriptors are built once and advanced by constant offsets (their
      // start-address field is in 16-byte units).
      auto issue_s = [&](int t, int ik) {
        const uint64_t da = sdesc_sw128(sbase + C::kQOff + t * C::kTileBytes, 16, 1024);
        const uint64_t db = sdesc_sw128(kv_smem(ik), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_w(tmem + C::col_s(t), da + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V: A = P_t from TMEM (8 columns per K step of 16), B = V
      // tile, MN-major (d contiguous): K step = 16 rows = 2048 bytes, the
      // next 64 columns of d are one chunk (16 KiB) away.
      auto issue_pv = [&](int t, int iv, uint32_t acc) {
        const uint64_t dv = sdesc_sw128(kv_smem(iv), C::kChunkBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts_w(tmem + C::col_o(t), tmem + C::col_p(t) + 8 * kk, dv + ((kk * 2048) >> 4),
                   idesc_pv, kk > 0 ? 1u : acc);
      };
      if (!mbar_wait_warp(b.q_full, 0, wc, kWaitQFull)) goto mma_end;
      if (!mbar_wait_warp(kv_full(0), kv_parity(0), wc, kWaitKvFull)) goto mma_end;
      tc_fence_after();
      for (int t = 0; t < 2; ++t) {
        if (n_t[t] > 0) {
          issue_s(t, 0);
          mma_commit_w(b.s_full[t]);
        }
      }
      mma_commit_w(kv_empty(0));
      for (int j = 0; j < nt; ++j) {
        const int iv = 2 * j + 1;
        const int ikn = 2 * j + 2;
        if (!mbar_wait_warp(kv_full(iv), kv_parity(iv), wc, kWaitKvFull)) goto mma_end;
        if (j < n_t[0]) {
          if (!mbar_wait_warp(b.p_full[0], j & 1, wc, kWaitPFull)) goto mma_end;
          tc_fence_after();
          issue_pv(0, iv, j > 0 ? 1u : 0u);
          if (j == n_t[0] - 1) mma_commit_w(b.o_full[0]);
        }
        if (j + 1 < nt) {
          if (!mbar_wait_warp(kv_full(ikn), kv_parity(ikn), wc, kWaitKvFull)) goto mma_end;
          tc_fence_after();
        }
        if (j + 1 < n_t[0]) {
          issue_s(0, ikn);
          mma_commit_w(b.s_full[0]);
        }
        if (j < n_t[1]) {
          if (!mbar_wait_warp(b.p_full[1], j & 1, wc, kWaitPFull)) goto mma_end;
          tc_fence_after();
          issue_pv(1, iv, j > 0 ? 1u : 0u);
          if (j == n_t[1] - 1) mma_commit_w(b.o_full[1]);
        }
        mma_commit_w(kv_empty(iv));
        if (j + 1 < n_t[1]) {
          issue_s(1, ikn);
          mma_commit_w(b.s_full[1]);
        }
        if (j + 1 < nt) mma_commit_w(kv_empty(ikn));
      }
    mma_end:
      // No MMA may still be running when TMEM is released.
      mma_commit_w(b.mma_done);
      mbar_wait_drain(b.mma_done, 0, args.wait_budget);
    }
    __syncwarp();
  } else if (warp == kLoadWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ TMA producer
    // Converged warp; one elected lane issues each copy.
    {
      int issued = 0;
      uint32_t qbytes = 0;
      for (int t = 0; t < 2; ++t) qbytes += n_t[t] > 0 ? C::kTileBytes : 0;
      mbar_arrive_expect_tx_w(b.q_full, qbytes);
      for (int t = 0; t < 2; ++t) {
        if (n_t[t] == 0) continue;
        for (int cc = 0; cc < C::kChunks; ++cc)
          tma_load_3d_w(sbase + C::kQOff + t * C::kTileBytes + cc * C::kChunkBytes, &tm_q,
                        b.q_full, cc * 64, q0 + t * kBM, bh);
      }
      for (int i = 0; i < 2 * nt; ++i) {
        const int s = i % C::kStages;
        const int r = i / C::kStages;
        if (r > 0 && !mbar_wait_warp(b.kv_empty0 + 8u * s, (r - 1) & 1, wc, kWaitKvEmpty)) break;
        const uint32_t full = b.kv_full0 + 8u * s;
        mbar_arrive_expect_tx_w(full, C::kTileBytes);
        const CUtensorMap* tm = (i & 1) ? &tm_v : &tm_k;
        const uint32_t dst = sbase + C::kKvOff + s * C::kTileBytes;
        for (int cc = 0; cc < C::kChunks; ++cc)
          tma_load_3d_w(dst + cc * C::kChunkBytes, tm, full, cc * 64, (i >> 1) * kBN, bh);
        issued = i + 1;
      }
      // Every copy this warp started must have landed before the CTA exits.
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait_drain(b.kv_full0 + 8u * (i % C::kStages), (i / C::kStages) & 1,
                        args.wait_budget);
      mbar_wait_drain(b.q_full, 0, args.wait_budget);
    }
    __syncwarp();
  } else {
    // warps 10-11: no work; they only hand their registers back.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD, bool CAUSAL>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<HD>;
  auto kern = fwd_kernel<HD, CAUSAL>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel is only valid for this launch size.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  const int num_pairs = (a.N + 2 * kBM - 1) / (2 * kBM);
  const dim3 grid(static_cast<unsigned>(num_pairs * a.BH));
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& a,
                       cudaStream_t stream) {
  if (d == 64) {
    return causal ? launch_fwd_t<64, true>(tq, tk, tv, to, a, stream)
                  : launch_fwd_t<64, false>(tq, tk, tv, to, a, stream);
  }
  return causal ? launch_fwd_t<128, true>(tq, tk, tv, to, a, stream)
                : launch_fwd_t<128, false>(tq, tk, tv, to, a, stream);
}

}  // namespace fattn
