// Main backward kernel of exact attention on sm_103a.
//
// Recomputation backward ("6.1 FlashAttention V1详解" §6.1-6.2): a work item
// is a 128-row K/V tile j of one (batch, head); it walks the 128-row Q tiles
// i (i >= j when causal).  Per step, with the kv rows on TMEM lanes:
//   S^T  = K_j Q_i^T                    (tcgen05, fp32 in TMEM)
//   P^T  = 2^(S^T*scale*log2e - L_i*log2e)    (one thread per kv row and query half; bf16 back to TMEM)
//   dP^T = V_j dO_i^T                   (tcgen05)
//   dS^T = P^T o (dP^T - D_i)           (bf16 to TMEM and, as dS, to shared memory)
//   dV_j += P^T dO_i                    (tcgen05, accumulator in TMEM)
//   dQ_i  = dS K_j                      (tcgen05) -> fp32 reduce-adds into dq_accum
//   dK_j += dS^T Q_i                    (tcgen05, issued after dQ: see below)
// At the end of an item dK_j * scale and dV_j are stored as bf16.  dQ = scale *
// dq_accum is converted by a separate kernel.  The dQ and dK formulas follow
// from S = scale Q K^T by the chain rule (the pages stop at dS).
//
// Persistent ("FlashAttention v1～v4" v4 §4 scheduling): one CTA per SM walks
// items numbered heaviest first (causal: small j has the most Q tiles) in
// L2-sized head sections and dealt in snake order (see bwd_item in
// fattn_sched.h).  The Q/dO ring and every per-step barrier run on one
// step counter across items, so the next item's first loads and MMAs start
// while this item's last dQ tile drains and its dK/dV are written out: V is
// released after the item's last dP^T, K after its last dQ, and dK/dV go from
// TMEM to global memory through the warps' own parts of the dS buffer (the
// K/V tiles are already being refilled), in whole 128-byte row segments.
//
// The global reduce-adds of dQ are capped per SM (about 25 bytes/cycle
// measured on GB300, whatever the path), so a 64 KiB dQ tile costs ~2600
// cycles, longer than the step's five MMAs (~2560 cycles at the tensor
// rate).  They are therefore taken off the critical path: a parking warpgroup
// copies the fp32 dQ tile out of TMEM into the Q/dO shared-memory stage that
// the step has just finished with (64 KiB at d = 128, 32 KiB at d = 64:
// exactly a dQ tile), in the 32 x 32 swizzled boxes of the accumulator's
// tensor map, which frees TMEM for the next dP^T; a reduce warp streams the
// boxes out with TMA reduce-adds and only then hands the stage back to the
// loader.  The compute warps never wait for either.
//
// Warps: 0-7 compute, as two warpgroups that split the 128 query columns of
// every key row (P and dS are elementwise, so the halves never exchange
// anything); 8 TMEM allocation + MMA issue; 9 TMA producer; 10 dQ reduce;
// 11 idle; 12-15 dQ parking.
// TMEM (512 columns): A [0,128) holds S^T, then P^T and dS^T; B [128,256)
// holds dP^T, then dQ ([128,128+d)).  Each warpgroup packs its 64 bf16
// values of P^T (32 columns) into the first half of the 64 fp32 columns of
// S^T it read itself (query 0-63 -> [0,32), query 64-127 -> [64,96)) and
// its dS^T into the second half ([32,64), [96,128)), never into columns the
// other warpgroup may still be reading.  dV at [256,256+d), dK at
// [256+d,256+2d).
// With dS^T out of B, dQ can be computed into B as soon as dS is complete,
// before dK: the chain dS -> dQ -> dQ parked -> next dP^T -> next dS sets the
// pace of a step (a clock64 trace: ~4600 cycles against 2560 of MMA), and dK
// now runs while dQ is being parked (measured on GB300: whole backward 645-647
// -> 622-626 us on B = 2, H = 32, N = 4096 causal, 2-3 % on the other
// shapes).  With dQ in B, the next S^T can be computed into A while the dQ
// rows are being read out.
#include "fattn_internal.h"
#include "fattn_ptx.cuh"
#include "fattn_sched.h"

namespace fattn {

namespace {

constexpr int kTile = 128;     // rows per Q tile and per K/V tile
constexpr int kThreads = 512;
constexpr int kComputeThreads = 256;
constexpr int kParkThreads = 128;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kReduceWarp = 10;
constexpr int kParkWarp0 = 12;
// Register split: the kernel launches with kLaunchRegs per thread (512 x 128 =
// 65,536); the compute warpgroups grow to kComputeRegs, the parking warpgroup
// sets kParkRegs (two 32-column TMEM loads in flight) and the control
// warpgroup (warps 8-11) shrinks to kCtrlRegs: 256 x 176 + 128 x 88 + 128 x 72
// = 65,536, exactly the launch total, so setmaxnreg.inc can always complete.
constexpr int kLaunchRegs = 128;
constexpr int kComputeRegs = 176;
constexpr int kParkRegs = 88;
constexpr int kCtrlRegs = 72;
static_assert(256 * kComputeRegs + 128 * kParkRegs + 128 * kCtrlRegs == kThreads * kLaunchRegs,
              "register split");
constexpr uint32_t kColA = 0, kColB = 128, kColDV = 256;

template <int HD>
struct BwdCfg {
  static constexpr int kChunks = HD / 64;
  static constexpr int kChunkBytes = kTile * 128;   // 128 rows x 128 bytes
  static constexpr int kTileBytes = kTile * HD * 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kStageOff = 2 * kTileBytes;  // stage s: Q_i then dO_i
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kDsOff = kStageOff + 2 * kStageBytes;
  static constexpr int kDsBytes = kTile * kTile * 2;
  static constexpr int kLdOff = kDsOff + kDsBytes;  // stage s: L2[128], D[128]
  static constexpr int kBarOff = kLdOff + 2 * 1024;
  static constexpr int kNumBars = 23;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16;
  static constexpr uint32_t kColDK = kColDV + HD;
  // The two K/V tile slots swap roles every item (which = 0: K, 1: V), so the
  // next item's K can land where this item's V was, one step before the end.
  __device__ static constexpr int kv_off(int m, int which) {
    return ((m ^ which) & 1) ? kVOff : kKOff;
  }
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Barrier indices.
enum : int {
  kBarKFull = 0,   // K_j landed (phase = item parity)
  kBarQFull = 1,   // +stage: Q_i and the L / D vectors landed
  kBarQEmpty = 3,  // +stage: Q_i's half of the stage is free again
  kBarSFull = 5,
  kBarDpFull = 6,
  kBarPFull = 7,
  kBarDsFull = 8,
  kBarDqFull = 9,
  kBarDqEmpty = 10,  // + (step & 1) via dq_empty(): dQ of the step parked
  kBarDkvFull = 11,
  kBarMmaDone = 12,
  kBarDoFull = 13,   // +stage: dO_i landed
  kBarDoEmpty = 15,  // +stage: dO_i's half of the stage is free again
  kBarVFull = 17,    // V_j landed
  kBarKEmpty = 18,   // the item's last MMA reading K_j has completed
  kBarVEmpty = 19,   // the item's last MMA reading V_j has completed
  kBarDkvEmpty = 20, // dK_j / dV_j have been read out of TMEM
  kBarDqEmpty1 = 21, // dQ-parked of the steps that use stage 1
  kBarDkDone = 22,   // the step's dK MMA (the last reader of Q_i) has completed
                     // (phase = step parity)
};

// dQ-parked barrier of a step: one per Q/dO stage, so that each completes
// once every two steps.  Parking step + 2 needs the stage that the reduce
// warp hands back after reading step's dQ, so the parking can be at most one
// phase of a stage's barrier ahead of any waiter, however long the reduce
// warp takes: a parity wait never confuses two phases.
__device__ __forceinline__ int dq_empty(uint32_t step) {
  return (step & 1) ? kBarDqEmpty1 : kBarDqEmpty;
}

// The Q tile that step it of item w visits (see BwdItem).
template <bool CAUSAL>
__device__ __forceinline__ int qtile(const BwdItem& w, int it, int n_tiles) {
  if constexpr (CAUSAL) {
    return w.i0 + it;
  } else {
    const int i = it + w.rot;
    return i >= n_tiles ? i - n_tiles : i;
  }
}

// The m-th work item of this CTA (false past the last one); see bwd_item.
template <bool CAUSAL>
__device__ __forceinline__ bool get_bwd_item(int m, int n_tiles, const BwdArgs& a, BwdItem& w) {
  return bwd_item<CAUSAL>(m, n_tiles, a, static_cast<int>(gridDim.x),
                          static_cast<int>(blockIdx.x), w);
}

template <int HD, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const __grid_constant__ CUtensorMap tm_dqacc,
               const __grid_constant__ BwdArgs args) {
  using C = BwdCfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  // The 128-byte swizzle needs 1024-byte aligned tiles.  The budget leaves no
  // room to realign, so a misaligned base is reported instead of used.
  if (sbase & 1023u) {
    if (threadIdx.x == 0 && atomicCAS(&args.status->code, 0u, 2u) == 0u) args.status->where = 100;
    return;
  }
  auto bar = [&](int i) { return sbase + C::kBarOff + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;
  const int n_tiles = (N + kTile - 1) / kTile;
  const int pitch = n_tiles * kTile;

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarKFull), 1);
    mbar_init(bar(kBarVFull), 1);
    mbar_init(bar(kBarKEmpty), 1);
    mbar_init(bar(kBarVEmpty), 1);
    mbar_init(bar(kBarDkvEmpty), kComputeThreads);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
      mbar_init(bar(kBarDoFull + s), 1);
      mbar_init(bar(kBarDoEmpty + s), 1);
    }
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarDpFull), 1);
    mbar_init(bar(kBarPFull), kComputeThreads);
    mbar_init(bar(kBarDsFull), kComputeThreads);
    mbar_init(bar(kBarDqFull), 1);
    mbar_init(bar(kBarDqEmpty), kParkThreads);
    mbar_init(bar(kBarDqEmpty1), kParkThreads);
    mbar_init(bar(kBarDkvFull), 1);
    mbar_init(bar(kBarDkDone), 1);
    mbar_init(bar(kBarMmaDone), 1);
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
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dqacc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtx wc{args.wait_budget, reinterpret_cast<volatile uint32_t*>(&misc[1]), args.status};

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kComputeRegs));
    // ================================================================ compute
    const int half = warp >> 2;              // query columns [64*half, 64*half + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;            // kv row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tA = tmem + lane_off + kColA;
    const uint32_t tB = tmem + lane_off + kColB;
    const uint64_t c2 = splat2(args.scale_log2);
    const uint32_t ds_base = sbase + C::kDsOff;
    const int col0 = 64 * half;
    bool ok = true;
    uint32_t step = 0;                       // steps done by this CTA (all items)
    BwdItem w;
    for (int m = 0; ok && get_bwd_item<CAUSAL>(m, n_tiles, args, w); ++m) {
      const int kv0 = w.j * kTile;
      const int kv = kv0 + r;
      const bool kv_valid = kv < N;
      for (int it = 0; it < w.n_it; ++it, ++step) {
        const int i = qtile<CAUSAL>(w, it, n_tiles);
        const int q0 = i * kTile;
        const int s = step & 1;
        const uint32_t ph = step & 1;
        const uint32_t* nl2s =
            reinterpret_cast<const uint32_t*>(smem + C::kLdOff + s * 1024) + col0;
        const uint32_t* ds_vec = nl2s + 128;
        dcheck(in_range(smem_u32(nl2s), 256, sbase + C::kLdOff, sbase + C::kBarOff) &&
                   in_range(smem_u32(ds_vec), 256, sbase + C::kLdOff, sbase + C::kBarOff),
               args.status, 402);
        // ---- P^T = 2^(S^T c - L2) (masked), this half's 64 query columns
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSFull), ph, wc, kWaitSFull));
        if (!ok) break;
        tc_fence_after();
        uint32_t p0[32], p1[32];
        tmem_ld32(tA + col0, p0);
        tmem_ld32(tA + col0 + 32, p1);
        tmem_ld_wait32(p0);
        reg_fence32(p1);
        uint32_t* pv[2] = {p0, p1};
        const bool diag = CAUSAL && q0 == kv0;
        // Only the diagonal tile and a K/V tile that runs past N need masks
        // (warp-uniform test); padded query columns already get exponent -inf.
        const bool need_mask = diag || kv0 + kTile > N;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            // nl2 = -L*log2(e) per query column (-inf past N)
            const uint4 l4 = *reinterpret_cast<const uint4*>(nl2s + g * 32 + e);
            uint32_t x[4];
            unpack2(ffma2(pack2(pv[g][e], pv[g][e + 1]), c2, pack2(l4.x, l4.y)), x[0], x[1]);
            unpack2(ffma2(pack2(pv[g][e + 2], pv[g][e + 3]), c2, pack2(l4.z, l4.w)), x[2], x[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) pv[g][e + u] = __float_as_uint(ex2_approx(__uint_as_float(x[u])));
          }
          if (need_mask) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int col = col0 + g * 32 + e;
              if (!kv_valid || (diag && col < r)) pv[g][e] = 0u;
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(pv[g][2 * e]), __uint_as_float(pv[g][2 * e + 1]));
          tmem_st16(tA + col0 + 16 * g, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull));
        // ---- dS^T = P^T o (dP^T - D)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarDpFull), ph, wc, kWaitDpFull));
        if (!ok) break;
        tc_fence_after();
        uint32_t dp0[32], dp1[32];
        tmem_ld32(tB + col0, dp0);
        tmem_ld32(tB + col0 + 32, dp1);
        tmem_ld_wait32(dp0);
        reg_fence32(dp1);
        uint32_t* dpv[2] = {dp0, dp1};
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const uint4 d4 = *reinterpret_cast<const uint4*>(ds_vec + g * 32 + e);
            uint32_t y[4];
            unpack2(fmul2(pack2(pv[g][e], pv[g][e + 1]),
                          fsub2(pack2(dpv[g][e], dpv[g][e + 1]), pack2(d4.x, d4.y))),
                    y[0], y[1]);
            unpack2(fmul2(pack2(pv[g][e + 2], pv[g][e + 3]),
                          fsub2(pack2(dpv[g][e + 2], dpv[g][e + 3]), pack2(d4.z, d4.w))),
                    y[2], y[3]);
            pk[e / 2] = pack_bf16x2(__uint_as_float(y[0]), __uint_as_float(y[1]));
            pk[e / 2 + 1] = pack_bf16x2(__uint_as_float(y[2]), __uint_as_float(y[3]));
          }
          tmem_st16(tA + col0 + 32 + 16 * g, pk);
          // dS row r, query columns [col0 + 32g, +32) = four 16-byte chunks of
          // the MN-major (query-contiguous) operand: 64-column atoms, 128-byte
          // swizzle inside each.
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const int c16 = (col0 >> 3) + g * 4 + qq;
            const uint32_t addr = ds_base + (c16 >> 3) * 16384 + r * 128 +
                                  (static_cast<uint32_t>((c16 & 7) ^ (r & 7)) << 4);
            if (dcheck(in_range(addr, 16, ds_base, ds_base + C::kDsBytes), args.status, 401))
              st_shared_v4(addr, pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(kBarDsFull));
      }
      if (!ok) break;
      // ---- item epilogue: warpgroup 0 writes dV_j, warpgroup 1 dK_j * scale,
      // as bf16.  Each warp stages its 32 rows, one 64-column chunk at a
      // time, in the part of the dS buffer that it writes dS into itself
      // (free from the item's last dQ MMA until its next dS), and reads them
      // back so that every store covers whole 128-byte row segments.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarDkvFull), m & 1, wc, kWaitOFull));
      if (!ok) break;
      tc_fence_after();
      {
        const uint32_t tsrc = tmem + lane_off + (half == 0 ? kColDV : C::kColDK);
        const float mul = half == 0 ? 1.f : args.scale;
        const uint32_t wbuf = ds_base + half * (kTile * 128) + wq * (32 * 128);
        uint16_t* const out = (half == 0 ? args.dv : args.dk) + static_cast<size_t>(w.bh) * N * HD;
#pragma unroll 1
        for (int cc = 0; cc < C::kChunks; ++cc) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t o[32];
            tmem_ld32(tsrc + 32 * (2 * cc + hh), o);
            tmem_ld_wait32(o);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * mul,
                                  __uint_as_float(o[2 * e + 1]) * mul);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const uint32_t c16 = hh * 4 + qq;
              const uint32_t a = wbuf + lane * 128 + ((c16 ^ (lane & 7)) << 4);
              if (dcheck(in_range(a, 16, ds_base, ds_base + C::kDsBytes), args.status, 403))
                st_shared_v4(a, pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
            }
          }
          __syncwarp();
          // 8 lanes per row, 4 rows per instruction.
#pragma unroll
          for (int rr = 0; rr < 32; rr += 4) {
            const int lr = rr + (lane >> 3);
            const uint32_t c16 = lane & 7;
            const uint4 v = ld_shared_v4(wbuf + lr * 128 + ((c16 ^ (lr & 7)) << 4));
            const int row = kv0 + wq * 32 + lr;
            const size_t o_idx = (static_cast<size_t>(w.bh) * N + row) * HD + cc * 64 + c16 * 8;
            if (row < N && dcheck(o_idx + 8 <= static_cast<size_t>(args.BH) * N * HD, args.status, 404))
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * HD + cc * 64 + c16 * 8) = v;
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarDkvEmpty));
    }
  } else if (warp == kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ MMA issue
    // The whole warp runs this (converged); one elected lane issues.
    {
      constexpr uint32_t idesc_kk = idesc_bf16_f32(kTile, kTile, false, false);
      constexpr uint32_t idesc_tm = idesc_bf16_f32(kTile, HD, false, true);
      constexpr uint32_t idesc_mm = idesc_bf16_f32(kTile, HD, true, true);
      const uint32_t sDs = sbase + C::kDsOff;
      auto sQ = [&](int s) { return sbase + C::kStageOff + s * C::kStageBytes; };
      auto sDo = [&](int s) { return sbase + C::kStageOff + s * C::kStageBytes + C::kTileBytes; };
      // D(128 x 128) = A(128 x HD) B(128 x HD)^T, both K-major (HD contiguous).
      auto mma_kmajor = [&](uint32_t d, uint32_t a, uint32_t b) {
        const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_w(d, da + off, db + off, idesc_kk, kk > 0 ? 1u : 0u);
        }
      };
      // D(128 x HD) (+)= A(tmem, 128 x 128) B, B MN-major (HD contiguous).
      // A's 16-query K steps sit at columns 8*kk for queries 0-63 and at
      // 64 + 8*(kk-4) for queries 64-127 (see the TMEM layout above).
      auto mma_tmem_a = [&](uint32_t d, uint32_t a_col, uint32_t b, uint32_t acc) {
        const uint64_t db = sdesc_sw128(b, C::kChunkBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_ts_w(d, tmem + a_col + (kk >> 2) * 64 + (kk & 3) * 8, db + ((kk * 2048) >> 4),
                   idesc_tm, kk > 0 ? 1u : acc);
      };
      auto qfull = [&](uint32_t g) {
        return mbar_wait_warp(bar(kBarQFull + (g & 1)), (g >> 1) & 1, wc, kWaitKvFull);
      };
      auto dofull = [&](uint32_t g) {
        return mbar_wait_warp(bar(kBarDoFull + (g & 1)), (g >> 1) & 1, wc, kWaitKvFull);
      };
      uint32_t step = 0;                     // steps issued by this CTA (all items)
      BwdItem w;
      for (int m = 0; get_bwd_item<CAUSAL>(m, n_tiles, args, w); ++m) {
        const int n_it = w.n_it;
        const uint32_t s0 = step & 1;
        const uint32_t sK = sbase + C::kv_off(m, 0), sV = sbase + C::kv_off(m, 1);
        // First S^T / dP^T of the item.  A is free (the previous item's last
        // dV, which read P^T there, was issued before); B still holds the
        // previous item's last dQ until the compute warps have parked it.
        if (!mbar_wait_warp(bar(kBarKFull), m & 1, wc, kWaitKvFull)) goto mma_end;
        if (!qfull(step)) goto mma_end;
        tc_fence_after();
        mma_kmajor(tmem + kColA, sK, sQ(s0));   // S^T
        mma_commit_w(bar(kBarSFull));
        if (m > 0 &&
            !mbar_wait_warp(bar(dq_empty(step - 1)), ((step - 1) >> 1) & 1, wc, kWaitDqEmpty))
          goto mma_end;
        if (!mbar_wait_warp(bar(kBarVFull), m & 1, wc, kWaitKvFull)) goto mma_end;
        if (!dofull(step)) goto mma_end;
        tc_fence_after();
        mma_kmajor(tmem + kColB, sV, sDo(s0));  // dP^T
        mma_commit_w(bar(kBarDpFull));
        if (n_it == 1) mma_commit_w(bar(kBarVEmpty));   // V_j's last reader issued
        for (int it = 0; it < n_it; ++it, ++step) {
          const int s = step & 1;
          const uint32_t ph = step & 1;
          const uint32_t acc = it > 0 ? 1u : 0u;
          if (!mbar_wait_warp(bar(kBarPFull), ph, wc, kWaitPFull)) goto mma_end;
          // The first dV / dK of an item overwrite the accumulators: the
          // previous item's must have been read out.
          if (it == 0 && m > 0 &&
              !mbar_wait_warp(bar(kBarDkvEmpty), (m - 1) & 1, wc, kWaitOFull))
            goto mma_end;
          tc_fence_after();
          mma_tmem_a(tmem + kColDV, kColA, sDo(s), acc);           // dV += P^T dO
          if (!mbar_wait_warp(bar(kBarDsFull), ph, wc, kWaitDsFull)) goto mma_end;
          tc_fence_after();
          // dQ = dS K into B first (the compute warps have read dP^T out of
          // it), so that its parking overlaps the dK product: A = dS (q
          // contiguous, MN-major), B = K (HD contiguous).
          {
            const uint64_t dds = sdesc_sw128(sDs, 16384, 1024);
            const uint64_t dk = sdesc_sw128(sK, C::kChunkBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              const uint32_t off = (kk * 2048) >> 4;
              mma_ss_w(tmem + kColB, dds + off, dk + off, idesc_mm, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit_w(bar(kBarDqFull));
          mma_tmem_a(tmem + C::kColDK, kColA + 32, sQ(s), acc);    // dK += dS^T Q
          mma_commit_w(bar(kBarDkDone));
          if (it + 1 < n_it) {
            if (!qfull(step + 1)) goto mma_end;
            tc_fence_after();
            mma_kmajor(tmem + kColA, sK, sQ(s ^ 1));               // S^T (next), overlaps the dQ read-out
            mma_commit_w(bar(kBarSFull));
            if (!mbar_wait_warp(bar(dq_empty(step)), (step >> 1) & 1, wc, kWaitDqEmpty))
              goto mma_end;
            if (!dofull(step + 1)) goto mma_end;
            tc_fence_after();
            mma_kmajor(tmem + kColB, sV, sDo(s ^ 1));              // dP^T (next)
            mma_commit_w(bar(kBarDpFull));
            if (it + 2 == n_it) mma_commit_w(bar(kBarVEmpty));   // V_j's last reader issued
          } else {
            mma_commit_w(bar(kBarKEmpty));     // K_j's last reader (this dQ) issued
            mma_commit_w(bar(kBarDkvFull));    // dV_j / dK_j complete
          }
        }
      }
    mma_end:
      mma_commit_w(bar(kBarMmaDone));
      mbar_wait_drain(bar(kBarMmaDone), 0, args.wait_budget);
    }
    __syncwarp();
  } else if (warp == kLoadWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ TMA producer
    // Converged warp; one elected lane issues each copy.
    {
      // Each stage is refilled in two halves, as the reduce warp frees them:
      // Q_i with the L / D vectors (needed first, by S^T), then dO_i.  An
      // item's K_j is loaded once the previous item's last dP^T has
      // completed (into that item's V slot), its first Q_i / dO_i next, and
      // V_j once the previous item's last dQ has completed; all four were
      // prefetched into L2 while the previous item's last steps ran.
      uint32_t step = 0;                     // Q and dO loads issued (steps)
      uint32_t issued_q = 0, issued_do = 0;
      // Q_i and dO_i are read again by the other K/V tiles of the head; K_j
      // and V_j once per item.  With these policies and the accumulator's
      // (reduce warp), measured on GB300, B = 2, H = 32, N = 4096 causal:
      // DRAM 707 -> 670 MB per launch, the whole backward 622-624 -> 616-617 us.
      const uint64_t pol_qdo = l2_evict_last_policy();
      const uint64_t pol_kv = l2_evict_first_policy();
      int items_v = 0, items_k = 0;
      BwdItem w;
      bool ok = true;
      // Q_i, the L / D vectors and dO_i of the CTA's next step into its stage.
      auto load_step = [&](const BwdItem& wi, int it) -> bool {
        const int s = step & 1;
        const uint32_t rnd = step >> 1;
        const int q0 = qtile<CAUSAL>(wi, it, n_tiles) * kTile;
        const uint32_t dst = sbase + C::kStageOff + s * C::kStageBytes;
        if (rnd > 0 && !mbar_wait_warp(bar(kBarQEmpty + s), (rnd - 1) & 1, wc, kWaitKvEmpty))
          return false;
        const uint32_t qf = bar(kBarQFull + s);
        mbar_arrive_expect_tx_w(qf, C::kTileBytes + 1024);
        for (int cc = 0; cc < C::kChunks; ++cc)
          tma_load_3d_hint_w(dst + cc * C::kChunkBytes, &tm_q, qf, cc * 64, q0, wi.bh, pol_qdo);
        const size_t vec = static_cast<size_t>(wi.bh) * pitch + q0;
        dcheck(vec + 128 <= static_cast<size_t>(args.BH) * pitch, args.status, 406);
        bulk_load_1d_w(sbase + C::kLdOff + s * 1024, args.L2 + vec, 512, qf);
        bulk_load_1d_w(sbase + C::kLdOff + s * 1024 + 512, args.D + vec, 512, qf);
        issued_q = step + 1;
        if (rnd > 0 && !mbar_wait_warp(bar(kBarDoEmpty + s), (rnd - 1) & 1, wc, kWaitKvEmpty))
          return false;
        const uint32_t df = bar(kBarDoFull + s);
        mbar_arrive_expect_tx_w(df, C::kTileBytes);
        for (int cc = 0; cc < C::kChunks; ++cc)
          tma_load_3d_hint_w(dst + C::kTileBytes + cc * C::kChunkBytes, &tm_do, df, cc * 64, q0,
                             wi.bh, pol_qdo);
        issued_do = step + 1;
        ++step;
        return true;
      };
      for (int m = 0; ok && get_bwd_item<CAUSAL>(m, n_tiles, args, w); ++m) {
        const int kv0 = w.j * kTile;
        // K_j goes where the previous item's V was, V_j where its K was.
        if (m > 0 && !mbar_wait_warp(bar(kBarVEmpty), (m - 1) & 1, wc, kWaitKvEmpty)) break;
        mbar_arrive_expect_tx_w(bar(kBarKFull), C::kTileBytes);
        for (int cc = 0; cc < C::kChunks; ++cc)
          tma_load_3d_hint_w(sbase + C::kv_off(m, 0) + cc * C::kChunkBytes, &tm_k,
                             bar(kBarKFull), cc * 64, kv0, w.bh, pol_kv);
        items_k = m + 1;
        if (!load_step(w, 0)) break;
        if (m > 0 && !mbar_wait_warp(bar(kBarKEmpty), (m - 1) & 1, wc, kWaitKvEmpty)) break;
        mbar_arrive_expect_tx_w(bar(kBarVFull), C::kTileBytes);
        for (int cc = 0; cc < C::kChunks; ++cc)
          tma_load_3d_hint_w(sbase + C::kv_off(m, 1) + cc * C::kChunkBytes, &tm_v,
                             bar(kBarVFull), cc * 64, kv0, w.bh, pol_kv);
        items_v = m + 1;
        for (int it = 1; it < w.n_it && ok; ++it) ok = load_step(w, it);
        BwdItem wn;
        if (ok && get_bwd_item<CAUSAL>(m + 1, n_tiles, args, wn)) {
          for (int cc = 0; cc < C::kChunks; ++cc) {
            tma_prefetch_l2_3d_w(&tm_k, cc * 64, wn.j * kTile, wn.bh);
            tma_prefetch_l2_3d_w(&tm_v, cc * 64, wn.j * kTile, wn.bh);
            tma_prefetch_l2_3d_w(&tm_q, cc * 64, qtile<CAUSAL>(wn, 0, n_tiles) * kTile, wn.bh);
            tma_prefetch_l2_3d_w(&tm_do, cc * 64, qtile<CAUSAL>(wn, 0, n_tiles) * kTile, wn.bh);
          }
        }
      }
      // Every copy this warp started must have landed before the CTA exits.
      for (uint32_t g = issued_q > 2 ? issued_q - 2 : 0; g < issued_q; ++g)
        mbar_wait_drain(bar(kBarQFull + (g & 1)), (g >> 1) & 1, args.wait_budget);
      for (uint32_t g = issued_do > 2 ? issued_do - 2 : 0; g < issued_do; ++g)
        mbar_wait_drain(bar(kBarDoFull + (g & 1)), (g >> 1) & 1, args.wait_budget);
      if (items_v > 0) mbar_wait_drain(bar(kBarVFull), (items_v - 1) & 1, args.wait_budget);
      if (items_k > 0) mbar_wait_drain(bar(kBarKFull), (items_k - 1) & 1, args.wait_budget);
    }
    __syncwarp();
  } else if (warp == kReduceWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ dQ reduce
    // For each step: once dQ_i has been parked in stage s, reduce-add its
    // boxes into the accumulator -- query rows 0-63 sit in the stage's Q
    // half, rows 64-127 in its dO half -- and hand each half back to the
    // loader as soon as the TMA engine has read it.  In deterministic mode
    // ("FlashAttention v1～v4" v4 §4) the adds into Q tile i wait for the
    // tile's counter to show that K/V tiles 0..j-1 have added theirs, and the
    // counter moves on to j+1 once this tile's adds have completed.
    uint32_t* const order = args.dq_order;
    // The accumulator lines take the reduce-adds of every K/V tile of the
    // head, then the conversion: keep them in L2.
    const uint64_t pol_acc = l2_evict_last_policy();
    bool ok = true;
    uint32_t step = 0;
    BwdItem w;
    for (int m = 0; ok && get_bwd_item<CAUSAL>(m, n_tiles, args, w); ++m) {
      for (int it = 0; it < w.n_it; ++it, ++step) {
        const int s = step & 1;
        const int qt = qtile<CAUSAL>(w, it, n_tiles);
        const int q0 = qt * kTile;
        const int bh = w.bh;
        ok = mbar_wait_warp(bar(dq_empty(step)), (step >> 1) & 1, wc, kWaitDqEmpty);
        if (!ok) break;
        uint32_t* const cnt =
            order != nullptr ? order + static_cast<size_t>(bh) * n_tiles + qt : nullptr;
        if (cnt != nullptr) {
          bool turn = true;
          if (lane == 0) {
            turn = counter_wait(cnt, static_cast<uint32_t>(w.j), wc, kWaitDqOrder);
            fence_proxy_async_global();
          }
          ok = __shfl_sync(0xffffffffu, turn ? 1 : 0, 0) != 0;
          if (!ok) break;
        }
        if (lane == 0) {
          // 8 KiB groups (two boxes), at most two in flight: the TMA engine
          // serves the stage's loads in between instead of behind a whole
          // 64 KiB reduce that drains at the per-SM reduce-add rate.
          const uint32_t stage = sbase + C::kStageOff + s * C::kStageBytes;
          for (int qb = 0; qb < 4; ++qb) {
#pragma unroll
            for (int ch = 0; ch < HD / 32; ch += 2) {
              if (q0 + qb * 32 < N) {
                tma_reduce_add_3d_hint(&tm_dqacc, stage + (qb * (HD / 32) + ch) * 4096, ch * 32,
                                       q0 + qb * 32, bh, pol_acc);
                tma_reduce_add_3d_hint(&tm_dqacc, stage + (qb * (HD / 32) + ch + 1) * 4096,
                                       (ch + 1) * 32, q0 + qb * 32, bh, pol_acc);
              }
              bulk_commit_group();
              bulk_wait_group_read1();
            }
            if (qb == 1 && cnt == nullptr) {
              bulk_wait_group_read0();
              mbar_arrive(bar(kBarQEmpty + s));   // rows 0-63 (the Q half) read
            }
          }
          bulk_wait_group_read0();
          if (cnt != nullptr) {
            // The next K/V tile's adds into this Q tile may start once these
            // have completed.  The stage goes back only after that: handed
            // back at once, the loader's next Q/dO copies queue on the TMA
            // engine ahead of the completion and delay the release that the
            // next K/V tile's CTA waits for (measured: ordered backward 0.968
            // vs 0.888 ms on the causal N = 4096 workload).
            bulk_wait_group0();
            fence_proxy_async_global();
            st_release_gpu(cnt, static_cast<uint32_t>(w.j) + 1u);
            mbar_arrive(bar(kBarQEmpty + s));
          }
          mbar_arrive(bar(kBarDoEmpty + s));      // rows 64-127 (the dO half) read
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  } else if (warp >= kParkWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kParkRegs));
    // ================================================================ dQ parking
    // For each step: dQ_i rows (TMEM lane = query row), all d columns -> the
    // Q/dO stage of the step, as 32 x 32 fp32 boxes with the 128-byte
    // swizzle.  Query rows 64-127 land in the stage's dO half (its readers,
    // dP^T and dV, completed before dQ), rows 0-63 in its Q half once the
    // step's dK MMA, issued after dQ, has completed too.
    const int wq = warp & 3;
    const uint32_t tB = tmem + (static_cast<uint32_t>(wq * 32) << 16) + kColB;
    bool ok = true;
    uint32_t step = 0;
    BwdItem w;
    for (int m = 0; ok && get_bwd_item<CAUSAL>(m, n_tiles, args, w); ++m) {
      for (int it = 0; it < w.n_it; ++it, ++step) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarDqFull), step & 1, wc, kWaitDqFull));
        // Query rows 0-63 go to the stage's Q half, which the step's dK MMA
        // (issued after dQ) may still be reading.
        if (ok && wq < 2)
          ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarDkDone), step & 1, wc, kWaitDqFull));
        if (!ok) break;
        tc_fence_after();
        const uint32_t stage = sbase + C::kStageOff + (step & 1) * C::kStageBytes;
#pragma unroll
        for (int ch = 0; ch < HD / 32; ch += 2) {
          uint32_t d0[32], d1[32];
          tmem_ld32(tB + 32 * ch, d0);
          tmem_ld32(tB + 32 * (ch + 1), d1);
          tmem_ld_wait32(d0);
          reg_fence32(d1);
          const uint32_t box0 = stage + (wq * (HD / 32) + ch) * 4096 + lane * 128;
          dcheck(in_range(box0, 4096 + 128, stage, stage + C::kStageBytes), args.status, 405);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const uint32_t sw = static_cast<uint32_t>(c4 ^ (lane & 7)) << 4;
            st_shared_v4(box0 + sw, d0[4 * c4], d0[4 * c4 + 1], d0[4 * c4 + 2], d0[4 * c4 + 3]);
            st_shared_v4(box0 + 4096 + sw, d1[4 * c4], d1[4 * c4 + 1], d1[4 * c4 + 2],
                         d1[4 * c4 + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(dq_empty(step)));
      }
    }
  } else {
    // warp 11: no work; it only hands its registers back.
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
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tacc, const BwdArgs& a,
                         cudaStream_t stream) {
  using C = BwdCfg<HD>;
  auto kern = bwd_kernel<HD, CAUSAL>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel is only valid for this launch size.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  int l2 = 0;
  if ((e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return e;
  // Persistent grid: one CTA per SM (at most one per work item).
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const long long items = static_cast<long long>(n_tiles) * a.BH;
  if (items >= 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(items < sms ? items : sms));
  BwdArgs ab = a;
  plan_bwd_schedule(ab, n_tiles, HD, CAUSAL, a.dq_order != nullptr, static_cast<int>(grid.x), l2);
  if (a.dq_order == nullptr) {
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tacc, ab);
    return cudaGetLastError();
  }
  // Ordered mode: a CTA waits for dQ adds of CTAs holding smaller K/V tiles,
  // so every CTA of the grid must be resident at once.  A cooperative launch
  // guarantees that (or fails up front) even when other work shares the GPU.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tacc, ab);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return e;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tacc, const BwdArgs& a, cudaStream_t stream) {
  if (d == 64) {
    return causal ? launch_bwd_t<64, true>(tq, tk, tv, tdo, tacc, a, stream)
                  : launch_bwd_t<64, false>(tq, tk, tv, tdo, tacc, a, stream);
  }
  return causal ? launch_bwd_t<128, true>(tq, tk, tv, tdo, tacc, a, stream)
                : launch_bwd_t<128, false>(tq, tk, tv, tdo, tacc, a, stream);
}

}  // namespace fattn
