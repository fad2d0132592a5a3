// Main backward kernel of exact attention on sm_103a, CTA-pair version
// (d = 128, any-order dQ).
//
// Same recomputation backward as fattn_bwd.cu ("6.1 FlashAttention V1详解"
// §6.1-6.2), with the five matrix products issued for a cluster of two CTAs
// on two SMs ("FlashAttention v1～v4" v4 §4: two CTAs cooperate on one MMA,
// each staging half of operand B, so the hardware sees an M = 256 tile; half
// of dS is exchanged through distributed shared memory and the dQ
// reductions are halved).  A work item is a unit of two K/V tiles of one
// (batch, head): tile 2u on CTA rank 0, tile 2u + 1 on rank 1, 256 keys.
// Per step (one 128-row Q tile) the leader (rank 0) issues, with
// tcgen05.mma.cta_group::2:
//   S^T  = K Q^T      M = 256 (each CTA its 128 keys), N = 128 queries,
//                     each CTA staging 64 query rows of Q (all d)
//   dP^T = V dO^T     likewise with V and dO
//   dV  += P^T dO     M = 256, A = P^T from each CTA's TMEM, N = d split:
//                     each CTA stages 64 of the d columns of dO (all queries)
//   dK  += dS^T Q     likewise with Q
//   dQ   = dS K       M = 128 (each CTA 64 query rows), K = all 256 keys of
//                     the unit, N = d split: each CTA stages 64 d columns of
//                     both K tiles; so dQ arrives summed over the unit's 256
//                     keys, 64 query rows per CTA
// and the CTAs run the same softmax-side work as the single-CTA kernel on
// their own 128 keys.  Each compute thread writes its key row's dS for the
// 64 queries of its half into the dS operand of the CTA that owns those
// query rows (its own, or the peer's through distributed shared memory).
// Per step and CTA the MMA operands move ~192 KiB through shared memory
// (256 KiB with one CTA per tile) and the fp32 dQ tile that is parked and
// reduce-added is 32 KiB (64 KiB).
//
// Warps (each CTA): 0-7 compute (two warpgroups splitting the 128 query
// columns of every key row), 8 TMEM allocation + (rank 0) MMA issue, 9 TMA
// producer, 10 dQ reduce, 11 (rank 1) relay to the leader, 12-15 dQ parking.
// TMEM (512 columns, allocated for the pair): [0,128) S^T, then P^T;
// [128,256) dP^T, then dS^T, then dQ in [128,192) (lane l < 64: query
// 64 rank + l, d [0,64); lane 64 + l: the same query, d [64,128)); dV
// [256,384); dK [384,512).
// Shared memory (per CTA): own K tile (K-major, the A operand of S^T), own V
// tile, K_Q (both K tiles of the unit, this CTA's 64 d columns: dQ's B), two
// stages of {Q_S, dO_S} (this CTA's 64 query rows, all d: S^T / dP^T's B;
// the stage later holds the parked fp32 dQ tile), one buffer of {Q_K, dO_V}
// (all 128 queries, this CTA's 64 d columns: dK / dV's B), dS_Q (256 keys x
// this CTA's 64 queries: dQ's A), the L / D vectors.
//
// Every operand a pair MMA reads must be in place in both CTAs before the
// leader issues it.  TMA loads of both CTAs complete on the leader's
// barriers (cp.async.bulk.tensor .cta_group::2); the leader's commits arrive
// on the barrier at the same offset in both CTAs (multicast).  Compute,
// parking and epilogue warps arrive only on barriers of their own CTA: on
// GB300 an arrival with cluster-scope release, or a cluster-scope proxy
// fence, costs ~600-1500 cycles in the issuing warp under load (measured),
// against ~10 for a CTA-scope one.  In the peer CTA, warp 11 relays each
// such phase to the leader with one relaxed arrival, in the order the leader
// consumes them.  The half of dS that the other CTA needs goes there with
// st.async, whose bytes complete on the receiving CTA's own barrier.  Every
// wait is bounded; a wait that runs out records FATTN_ERR_TIMEOUT and the
// CTA winds down, as in the single-CTA kernel.
#include "fattn_internal.h"
#include "fattn_ptx.cuh"
#include "fattn_sched.h"

namespace fattn {

namespace {

constexpr int kTile = 128;
constexpr int kHd = 128;
constexpr int kThreads = 512;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kReduceWarp = 10;
constexpr int kRelayWarp = 11;
constexpr int kParkWarp0 = 12;
// Register split as in the single-CTA kernel: 256 x 176 + 128 x 88 +
// 128 x 72 = 512 x 128.
constexpr int kLaunchRegs = 128;
constexpr int kComputeRegs = 176;
constexpr int kParkRegs = 88;
constexpr int kCtrlRegs = 72;
static_assert(256 * kComputeRegs + 128 * kParkRegs + 128 * kCtrlRegs == kThreads * kLaunchRegs,
              "register split");

constexpr uint32_t kColA = 0, kColB = 128, kColDV = 256, kColDK = 384;

// Shared-memory layout (bytes).
constexpr int kKaOff = 0;           // own K tile: 2 panels of 64 d columns x 128 rows
constexpr int kVOff = 32768;        // own V tile
constexpr int kKqOff = 65536;       // K_Q: keys 0-127 of the unit, then 128-255; 64 d columns
constexpr int kStageOff = 98304;    // 2 x 32 KiB: Q_S (2 panels x 64 rows), then dO_S
constexpr int kStageBytes = 32768;
constexpr int kQkOff = 163840;      // Q_K: 128 queries x this CTA's 64 d columns
constexpr int kDovOff = 180224;     // dO_V
constexpr int kDsqOff = 196608;     // dS_Q: 256 key rows x 64 queries
constexpr int kLdOff = 229376;      // 2 x 1 KiB: -L log2(e) [128], D [128]
constexpr int kBarOff = 231424;
constexpr int kNumBars = 36;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kMiscOff + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// Barriers.  The first two groups are used in the leader only: operands of
// its MMAs (TMA completions from both CTAs) and the peer's relayed phases;
// the others in both CTAs.
enum : int {
  kBKFull = 0,       // both own K tiles landed
  kBVFull = 1,
  kBKqFull = 2,
  kBQsFull = 3,      // +stage: Q_S of both CTAs
  kBDosFull = 5,     // +stage: dO_S of both CTAs
  kBQkFull = 7,      // Q_K of both CTAs
  kBDovFull = 8,     // dO_V of both CTAs
  kBPRemote = 9,     // --- relayed by the peer: its P^T is in TMEM
  kBDsRemote = 10,   // its dS^T is in TMEM (and its own half of dS_Q stored)
  kBDsqRemote = 11,  // the leader's half of dS has reached its dS_Q
  kBDqRemote = 12,   // +(step & 1): its dQ tile has been read out of TMEM
  kBDkvRemote = 14,  // its dK / dV are out of TMEM and stored
  kBPLocal = 15,     // --- both CTAs: local warps
  kBDsLocal = 16,    // 8 compute warps: dS^T in TMEM, own half of dS_Q stored
  kBDsqFull = 17,    // the 16 KiB of dS the other CTA sends (posted by compute warp 0)
  kBDqParked = 18,   // +(step & 1): 4 parking warps
  kBEpiDone = 20,    // 8 compute warps (K_Q free, dK / dV stored)
  kBSFull = 21,      // --- both CTAs: multicast commits of the leader
  kBDpFull = 22,
  kBDqFull = 23,
  kBDkvFull = 24,
  kBQkEmpty = 25,
  kBDovEmpty = 26,
  kBKEmpty = 27,
  kBVEmpty = 28,
  kBStageEmpty = 29, // +stage: the parked dQ has been read by the reduce-adds
  kBLdFull = 31,     // +stage: L / D vectors
  kBMmaDone = 33,
  kBDqRead = 34,     // +(step & 1): 4 parking warps have read dQ out of TMEM
};

__device__ __forceinline__ int dq_slot(uint32_t step) { return static_cast<int>(step & 1); }

template <bool CAUSAL>
__device__ __forceinline__ int qtile2(const BwdItem& w, int it, int n_tiles) {
  if constexpr (CAUSAL) {
    return w.i0 + it;
  } else {
    const int i = it + w.rot;
    return i >= n_tiles ? i - n_tiles : i;
  }
}

template <bool CAUSAL>
__device__ __forceinline__ bool get_item2(int m, int n_tiles, const BwdArgs& a, BwdItem& w) {
  return bwd2_item<CAUSAL>(m, n_tiles, a, static_cast<int>(gridDim.x >> 1),
                           static_cast<int>(blockIdx.x >> 1), w);
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q64,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_do64,
                const __grid_constant__ CUtensorMap tm_dqacc,
                const __grid_constant__ BwdArgs args) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rank = cluster_rank();
  auto bar = [&](int i) { return sbase + kBarOff + 8u * i; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  // The base is the same in both CTAs (same kernel, same dynamic size); a
  // misaligned one is reported by each CTA, and both still meet at the
  // cluster barriers below.
  const bool aligned = (sbase & 1023u) == 0;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;
  const int n_tiles = (N + kTile - 1) / kTile;
  const int pitch = n_tiles * kTile;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBQsFull + i), 1);
      mbar_init(bar(kBDosFull + i), 1);
      mbar_init(bar(kBDqRemote + i), 1);
      mbar_init(bar(kBDqParked + i), 4);
      mbar_init(bar(kBDqRead + i), 4);
      mbar_init(bar(kBStageEmpty + i), 1);
      mbar_init(bar(kBLdFull + i), 1);
    }
    for (int i : {kBKFull, kBVFull, kBKqFull, kBQkFull, kBDovFull, kBPRemote, kBDsRemote,
                  kBDsqRemote, kBDkvRemote, kBDsqFull, kBSFull, kBDpFull, kBDqFull, kBDkvFull,
                  kBQkEmpty, kBDovEmpty, kBKEmpty, kBVEmpty, kBMmaDone})
      mbar_init(bar(i), 1);
    mbar_init(bar(kBPLocal), 8);
    mbar_init(bar(kBDsLocal), 8);
    mbar_init(bar(kBEpiDone), 8);
    misc[1] = aligned ? 0u : 1u;
    if (!aligned && atomicCAS(&args.status->code, 0u, 2u) == 0u) args.status->where = 101;
    fence_barrier_init();
  }
  // Both CTAs' barriers exist before either CTA signals the other.
  cluster_sync_all();
  if (warp == kMmaWarp) {
    tmem_alloc_pair(smem_u32(&misc[0]), 512);
    tmem_relinquish_pair();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_q64);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_do64);
    tma_prefetch_desc(&tm_dqacc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtx wc{args.wait_budget, reinterpret_cast<volatile uint32_t*>(&misc[1]), args.status};
  auto lead = [&](int i) { return map_shared(bar(i), 0); };

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kComputeRegs));
    // ================================================================ compute
    const int half = warp >> 2;              // query columns [64*half, 64*half + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;            // key row of this CTA's tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tA = tmem + lane_off + kColA;
    const uint32_t tB = tmem + lane_off + kColB;
    const uint64_t c2 = splat2(args.scale_log2);
    // dS of query half `half` goes to the dS_Q operand of CTA `half`, at the
    // row of this key within the unit (rank 0's keys first).  The warpgroup
    // of this CTA's own half stores into its dS_Q directly; the other stages
    // its 128 rows in the step's Q_S buffer (read by S^T, which has completed
    // by then) and sends them to the other CTA with bulk copies, 4 KiB per
    // warp.
    const int ds_row = static_cast<int>(rank) * kTile + r;
    const bool ds_local = half == static_cast<int>(rank);
    const uint32_t peer = rank ^ 1u;
    const int col0 = 64 * half;
    bool ok = misc[1] == 0u;
    uint32_t step = 0;
    BwdItem w;
    for (int m = 0; ok && get_item2<CAUSAL>(m, n_tiles, args, w); ++m) {
      const int kv0 = (w.j + static_cast<int>(rank)) * kTile;
      const int kv = kv0 + r;
      const bool kv_valid = kv < N;
      for (int it = 0; it < w.n_it; ++it, ++step) {
        const int i = qtile2<CAUSAL>(w, it, n_tiles);
        const int q0 = i * kTile;
        const int s = step & 1;
        const uint32_t ph = step & 1;
        const uint32_t* nl2s =
            reinterpret_cast<const uint32_t*>(smem + kLdOff + s * 1024) + col0;
        const uint32_t* ds_vec = nl2s + 128;
        dcheck(in_range(smem_u32(nl2s), 256, sbase + kLdOff, sbase + kBarOff) &&
                   in_range(smem_u32(ds_vec), 256, sbase + kLdOff, sbase + kBarOff),
               args.status, 502);
        ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(kBLdFull + s), (step >> 1) & 1, wc,
                                                  kWaitQFull));
        if (!ok) break;
        // ---- P^T = 2^(S^T c - L2) (masked), this half's 64 query columns
        ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(kBSFull), ph, wc, kWaitSFull));
        if (!ok) break;
        tc_fence_after();
        uint32_t p0[32], p1[32];
        tmem_ld32(tA + col0, p0);
        tmem_ld32(tA + col0 + 32, p1);
        tmem_ld_wait32(p0);
        reg_fence32(p1);
        uint32_t* pv[2] = {p0, p1};
        // Masks only where some key of this tile lies after some query of the
        // Q tile (causal) or past N; padded query columns already get
        // exponent -inf.
        const bool need_mask = (CAUSAL && q0 < kv0 + kTile) || kv0 + kTile > N;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
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
              const int q = q0 + col0 + g * 32 + e;
              if (!kv_valid || (CAUSAL && q < kv)) pv[g][e] = 0u;
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
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBPLocal));
        // ---- dS^T = P^T o (dP^T - D)
        ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(kBDpFull), ph, wc, kWaitDpFull));
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
          tmem_st16(tB + col0 + 16 * g, pk);
          // dS row (key ds_row), queries [32g, 32g + 32) of this half: four
          // 16-byte chunks of the MN-major (query-contiguous) operand, with
          // the 128-byte swizzle.
          const uint32_t row_addr =
              ds_local ? sbase + kDsqOff + static_cast<uint32_t>(ds_row) * 128u
                       : sbase + kStageOff + s * kStageBytes + static_cast<uint32_t>(r) * 128u;
          dcheck(ds_local ? in_range(row_addr, 128, sbase + kDsqOff, sbase + kLdOff)
                          : in_range(row_addr, 128, sbase + kStageOff + s * kStageBytes,
                                     sbase + kStageOff + s * kStageBytes + 16384),
                 args.status, 501);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint32_t c16 = static_cast<uint32_t>(g * 4 + qq);
            st_shared_v4(row_addr + ((c16 ^ static_cast<uint32_t>(r & 7)) << 4), pk[4 * qq],
                         pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        if (!ds_local) {
          // This warp's 32 staged rows are rows 128 rank + 32 wq .. + 31 of
          // the other CTA's dS_Q, with the same swizzle (row & 7 == r & 7):
          // one 4 KiB bulk copy per warp, as soon as the warp has staged them.
          __syncwarp();
          if (lane == 0) {
            const uint32_t off = static_cast<uint32_t>(wq) * 4096u;
            bulk_copy_to_cluster(
                map_shared(sbase + kDsqOff + rank * (kTile * 128u) + off, peer),
                sbase + kStageOff + s * kStageBytes + off, 4096, map_shared(bar(kBDsqFull), peer));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kBDsLocal));
          // ... and warp 0 posts the 16 KiB that the other CTA's compute warps
          // send into this CTA's dS_Q for this step.
          if (warp == 0) mbar_arrive_expect_tx(bar(kBDsqFull), 16384);
        }
      }
      if (!ok) break;
      // ---- item epilogue: warpgroup 0 writes dV, warpgroup 1 dK * scale, as
      // bf16, staged per warp through this CTA's K_Q buffer (free from the
      // item's last dQ until the loader refills it after EpiDone), so that
      // every store covers whole 128-byte row segments.
      ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(kBDkvFull), m & 1, wc, kWaitOFull));
      if (!ok) break;
      tc_fence_after();
      {
        const uint32_t tsrc = tmem + lane_off + (half == 0 ? kColDV : kColDK);
        const float mul = half == 0 ? 1.f : args.scale;
        const uint32_t wbuf = sbase + kKqOff + half * 16384 + wq * 4096;
        uint16_t* const out = (half == 0 ? args.dv : args.dk) + static_cast<size_t>(w.bh) * N * kHd;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
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
              if (dcheck(in_range(a, 16, sbase + kKqOff, sbase + kStageOff), args.status, 503))
                st_shared_v4(a, pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
            }
          }
          __syncwarp();
#pragma unroll
          for (int rr = 0; rr < 32; rr += 4) {
            const int lr = rr + (lane >> 3);
            const uint32_t c16 = lane & 7;
            const uint4 v = ld_shared_v4(wbuf + lr * 128 + ((c16 ^ (lr & 7)) << 4));
            const int row = kv0 + wq * 32 + lr;
            const size_t o_idx = (static_cast<size_t>(w.bh) * N + row) * kHd + cc * 64 + c16 * 8;
            if (row < N && dcheck(o_idx + 8 <= static_cast<size_t>(args.BH) * N * kHd, args.status, 504))
              *reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * kHd + cc * 64 + c16 * 8) = v;
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBEpiDone));
    }
  } else if (warp == kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ MMA issue (leader)
    if (rank == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(256, kTile, false, false);
      constexpr uint32_t idesc_t = idesc_bf16_f32(256, kHd, false, true);
      constexpr uint32_t idesc_q = idesc_bf16_f32(128, kHd, true, true);
      auto stage = [&](int s) { return sbase + kStageOff + s * kStageBytes; };
      // D(256 x 128) = A(own 128 rows x d per CTA) B(64 rows x d per CTA)^T,
      // both K-major: A panels of 16 KiB (128 rows), B panels of 8 KiB.
      auto mma_sT = [&](uint32_t d, uint32_t a, uint32_t b) {
        const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(b, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint32_t oa = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          const uint32_t ob = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
          mma2_ss_w(d, da + oa, db + ob, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      // D(256 x d) (+)= A(TMEM, own 128 rows x 128 queries per CTA) B(128
      // queries x 64 d columns per CTA), B MN-major.  A's 16-query K steps
      // sit at columns 8*kk (queries 0-63) and 64 + 8*(kk-4) (64-127).
      auto mma_tA = [&](uint32_t d, uint32_t a_col, uint32_t b, uint32_t acc) {
        const uint64_t db = sdesc_sw128(b, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma2_ts_w(d, tmem + a_col + (kk >> 2) * 64 + (kk & 3) * 8, db + ((kk * 2048) >> 4),
                    idesc_t, kk > 0 ? 1u : acc);
      };
      // dQ(128 x d; 64 query rows per CTA) = dS_Q(256 keys x 64 queries per
      // CTA, MN-major) K_Q(256 keys x 64 d columns per CTA, MN-major).
      auto mma_dq = [&]() {
        const uint64_t da = sdesc_sw128(sbase + kDsqOff, 8192, 1024);
        const uint64_t db = sdesc_sw128(sbase + kKqOff, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < 2 * kTile / 16; ++kk)
          mma2_ss_w(tmem + kColB, da + ((kk * 2048) >> 4), db + ((kk * 2048) >> 4), idesc_q,
                    kk > 0 ? 1u : 0u);
      };
      auto wait = [&](int b, uint32_t parity, unsigned int site) {
        return mbar_wait_cl_warp(bar(b), parity, wc, site);
      };
      // A phase of both CTAs' warps: this CTA's own barrier, then the peer's
      // relayed one.
      auto wait2 = [&](int local, int remote, uint32_t parity, unsigned int site) {
        return wait(local, parity, site) && wait(remote, parity, site);
      };
      bool ok = misc[1] == 0u;
      uint32_t step = 0;
      BwdItem w;
      for (int m = 0; ok && get_item2<CAUSAL>(m, n_tiles, args, w); ++m) {
        const int n_it = w.n_it;
        const int s0 = step & 1;
        if (!(ok = wait(kBKFull, m & 1, kWaitKvFull))) break;
        if (!(ok = wait(kBQsFull + s0, (step >> 1) & 1, kWaitKvFull))) break;
        tc_fence_after();
        mma_sT(tmem + kColA, sbase + kKaOff, stage(s0));               // S^T
        mma2_commit_both_w(bar(kBSFull));
        if (n_it == 1) mma2_commit_both_w(bar(kBKEmpty));
        if (m > 0 && !(ok = wait2(kBDqRead + dq_slot(step - 1), kBDqRemote + dq_slot(step - 1),
                                  ((step - 1) >> 1) & 1, kWaitDqEmpty)))
          break;
        if (!(ok = wait(kBVFull, m & 1, kWaitKvFull))) break;
        if (!(ok = wait(kBDosFull + s0, (step >> 1) & 1, kWaitKvFull))) break;
        tc_fence_after();
        mma_sT(tmem + kColB, sbase + kVOff, stage(s0) + 16384);        // dP^T
        mma2_commit_both_w(bar(kBDpFull));
        if (n_it == 1) mma2_commit_both_w(bar(kBVEmpty));
        for (int it = 0; it < n_it; ++it, ++step) {
          const int s = step & 1;
          const uint32_t ph = step & 1;
          const uint32_t acc = it > 0 ? 1u : 0u;
          if (!(ok = wait2(kBPLocal, kBPRemote, ph, kWaitPFull))) break;
          if (it == 0 && m > 0 && !(ok = wait2(kBEpiDone, kBDkvRemote, (m - 1) & 1, kWaitOFull)))
            break;
          if (!(ok = wait(kBDovFull, ph, kWaitKvFull))) break;
          tc_fence_after();
          mma_tA(tmem + kColDV, kColA, sbase + kDovOff, acc);           // dV += P^T dO
          mma2_commit_both_w(bar(kBDovEmpty));
          if (!(ok = wait2(kBDsLocal, kBDsRemote, ph, kWaitDsFull))) break;
          if (!(ok = wait(kBQkFull, ph, kWaitKvFull))) break;
          tc_fence_after();
          mma_tA(tmem + kColDK, kColB, sbase + kQkOff, acc);            // dK += dS^T Q
          mma2_commit_both_w(bar(kBQkEmpty));
          if (it == 0 && !(ok = wait(kBKqFull, m & 1, kWaitKvFull))) break;
          if (!(ok = wait2(kBDsqFull, kBDsqRemote, ph, kWaitDsFull))) break;
          fence_proxy_async_smem();   // the dS rows st.async delivered, for the MMA
          tc_fence_after();
          mma_dq();                                                    // dQ = dS K (256 keys)
          mma2_commit_both_w(bar(kBDqFull));
          if (it + 1 < n_it) {
            // S^T of the next step (it overwrites P^T, read by the dV issued
            // before): after dK and dQ, which the critical chain dQ -> parked
            // -> next dP^T waits for (MMAs run in issue order; issued before
            // them it measured slower).
            if (!(ok = wait(kBQsFull + (s ^ 1), ((step + 1) >> 1) & 1, kWaitKvFull))) break;
            tc_fence_after();
            mma_sT(tmem + kColA, sbase + kKaOff, stage(s ^ 1));         // S^T (next)
            mma2_commit_both_w(bar(kBSFull));
            if (it + 2 == n_it) mma2_commit_both_w(bar(kBKEmpty));
            if (!(ok = wait2(kBDqRead + dq_slot(step), kBDqRemote + dq_slot(step),
                             (step >> 1) & 1, kWaitDqEmpty)))
              break;
            if (!(ok = wait(kBDosFull + (s ^ 1), ((step + 1) >> 1) & 1, kWaitKvFull))) break;
            tc_fence_after();
            mma_sT(tmem + kColB, sbase + kVOff, stage(s ^ 1) + 16384);  // dP^T (next)
            mma2_commit_both_w(bar(kBDpFull));
            if (it + 2 == n_it) mma2_commit_both_w(bar(kBVEmpty));
          } else {
            mma2_commit_both_w(bar(kBDkvFull));
          }
        }
      }
      mma2_commit_both_w(bar(kBMmaDone));
      mbar_drain_cl(bar(kBMmaDone), 0, args.wait_budget);
    }
    __syncwarp();
  } else if (warp == kLoadWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ TMA producer
    // Both CTAs load their own shared memory; the copies that feed the
    // leader's MMAs complete on the leader's barriers, whose expected byte
    // counts (both CTAs' share) the leader's producer posts.
    const bool leader = rank == 0;
    const int rk = static_cast<int>(rank);
    uint32_t step = 0;
    uint32_t issued = 0;                     // steps whose Q_S / dO_S / L / D were issued
    uint32_t dov_posted = 0, qk_posted = 0;  // steps whose dO_V / Q_K were issued
    int k_items = 0, v_items = 0, kq_items = 0;
    bool ok = misc[1] == 0u;
    auto wait = [&](int b, uint32_t parity) {
      return mbar_wait_cl_warp(bar(b), parity, wc, kWaitKvEmpty);
    };
    auto post = [&](int b, uint32_t bytes) {
      if (leader) mbar_arrive_expect_tx_w(bar(b), bytes);
    };
    auto load_step = [&](const BwdItem& wi, int it) -> bool {
      const int s = step & 1;
      const uint32_t rnd = step >> 1;
      const int q0 = qtile2<CAUSAL>(wi, it, n_tiles) * kTile;
      const uint32_t dst = sbase + kStageOff + s * kStageBytes;
      if (rnd > 0 && !wait(kBStageEmpty + s, (rnd - 1) & 1)) return false;
      post(kBQsFull + s, 2 * 16384);
      for (int cc = 0; cc < 2; ++cc)
        tma2_load_3d_w(dst + cc * 8192, &tm_q64, lead(kBQsFull + s), cc * 64, q0 + 64 * rk,
                       wi.bh);
      post(kBDosFull + s, 2 * 16384);
      for (int cc = 0; cc < 2; ++cc)
        tma2_load_3d_w(dst + 16384 + cc * 8192, &tm_do64, lead(kBDosFull + s), cc * 64,
                       q0 + 64 * rk, wi.bh);
      const uint32_t lf = bar(kBLdFull + s);
      mbar_arrive_expect_tx_w(lf, 1024);
      const size_t vec = static_cast<size_t>(wi.bh) * pitch + q0;
      dcheck(vec + 128 <= static_cast<size_t>(args.BH) * pitch, args.status, 506);
      bulk_load_1d_w(sbase + kLdOff + s * 1024, args.L2 + vec, 512, lf);
      bulk_load_1d_w(sbase + kLdOff + s * 1024 + 512, args.D + vec, 512, lf);
      issued = step + 1;
      if (step > 0 && !wait(kBDovEmpty, (step - 1) & 1)) return false;
      post(kBDovFull, 2 * 16384);
      tma2_load_3d_w(sbase + kDovOff, &tm_do, lead(kBDovFull), 64 * rk, q0, wi.bh);
      dov_posted = step + 1;
      if (step > 0 && !wait(kBQkEmpty, (step - 1) & 1)) return false;
      post(kBQkFull, 2 * 16384);
      tma2_load_3d_w(sbase + kQkOff, &tm_q, lead(kBQkFull), 64 * rk, q0, wi.bh);
      qk_posted = step + 1;
      ++step;
      return true;
    };
    // K_Q doubles as the staging buffer of the previous item's dK / dV
    // stores, so it is refilled only once those are out; the item's first
    // two steps' operands go first.
    auto load_kq = [&](const BwdItem& wi, int m) -> bool {
      if (m > 0 && !mbar_wait_cl_warp(bar(kBEpiDone), (m - 1) & 1, wc, kWaitOFull)) return false;
      post(kBKqFull, 2 * 32768);
      for (int hh = 0; hh < 2; ++hh)
        tma2_load_3d_w(sbase + kKqOff + hh * 16384, &tm_k, lead(kBKqFull), 64 * rk,
                       wi.j * kTile + hh * kTile, wi.bh);
      kq_items = m + 1;
      return true;
    };
    BwdItem w;
    for (int m = 0; ok && get_item2<CAUSAL>(m, n_tiles, args, w); ++m) {
      const int kv_own = (w.j + rk) * kTile;
      if (m > 0 && !(ok = wait(kBKEmpty, (m - 1) & 1))) break;
      post(kBKFull, 2 * 32768);
      for (int cc = 0; cc < 2; ++cc)
        tma2_load_3d_w(sbase + kKaOff + cc * 16384, &tm_k, lead(kBKFull), cc * 64, kv_own, w.bh);
      k_items = m + 1;
      if (!(ok = load_step(w, 0))) break;
      if (m > 0 && !(ok = wait(kBVEmpty, (m - 1) & 1))) break;
      post(kBVFull, 2 * 32768);
      for (int cc = 0; cc < 2; ++cc)
        tma2_load_3d_w(sbase + kVOff + cc * 16384, &tm_v, lead(kBVFull), cc * 64, kv_own, w.bh);
      v_items = m + 1;
      if (w.n_it > 1 && !(ok = load_step(w, 1))) break;
      if (!(ok = load_kq(w, m))) break;
      for (int it = 2; it < w.n_it && ok; ++it) ok = load_step(w, it);
      BwdItem wn;
      if (ok && get_item2<CAUSAL>(m + 1, n_tiles, args, wn)) {
        const int kvn = (wn.j + rk) * kTile;
        for (int cc = 0; cc < 2; ++cc) {
          tma_prefetch_l2_3d_w(&tm_k, cc * 64, kvn, wn.bh);
          tma_prefetch_l2_3d_w(&tm_v, cc * 64, kvn, wn.bh);
        }
      }
    }
    if (leader) {
      // Every copy of either CTA that completes on the leader's barriers must
      // have landed before the pair exits: drain the phases posted last.
      for (uint32_t g = issued > 2 ? issued - 2 : 0; g < issued; ++g) {
        mbar_drain_cl(bar(kBQsFull + (g & 1)), (g >> 1) & 1, args.wait_budget);
        mbar_drain_cl(bar(kBDosFull + (g & 1)), (g >> 1) & 1, args.wait_budget);
      }
      if (dov_posted > 0) mbar_drain_cl(bar(kBDovFull), (dov_posted - 1) & 1, args.wait_budget);
      if (qk_posted > 0) mbar_drain_cl(bar(kBQkFull), (qk_posted - 1) & 1, args.wait_budget);
      if (k_items > 0) mbar_drain_cl(bar(kBKFull), (k_items - 1) & 1, args.wait_budget);
      if (v_items > 0) mbar_drain_cl(bar(kBVFull), (v_items - 1) & 1, args.wait_budget);
      if (kq_items > 0) mbar_drain_cl(bar(kBKqFull), (kq_items - 1) & 1, args.wait_budget);
    } else if (!ok) {
      // The leader may have stopped posting: give this CTA's last copies
      // time to land before the pair exits (they finish within microseconds).
      for (int t = 0; t < 64; ++t) __nanosleep(1000);
    }
    for (uint32_t g = issued > 2 ? issued - 2 : 0; g < issued; ++g)
      mbar_drain_cl(bar(kBLdFull + (g & 1)), (g >> 1) & 1, args.wait_budget);
    __syncwarp();
  } else if (warp == kReduceWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ dQ reduce
    // This CTA's 64 query rows of the step's dQ tile, parked in its stage as
    // eight 32 x 32 fp32 boxes, are reduce-added into the accumulator; then
    // the stage goes back to the loader.
    bool ok = misc[1] == 0u;
    uint32_t step = 0;
    BwdItem w;
    for (int m = 0; ok && get_item2<CAUSAL>(m, n_tiles, args, w); ++m) {
      for (int it = 0; it < w.n_it; ++it, ++step) {
        const int s = step & 1;
        const int q0 = qtile2<CAUSAL>(w, it, n_tiles) * kTile + 64 * static_cast<int>(rank);
        ok = mbar_wait_cl_warp(bar(kBDqParked + dq_slot(step)), (step >> 1) & 1, wc, kWaitDqEmpty);
        if (!ok) break;
        if (lane == 0) {
          const uint32_t stg = sbase + kStageOff + s * kStageBytes;
          for (int qb = 0; qb < 2; ++qb) {
#pragma unroll
            for (int db = 0; db < 4; db += 2) {
              if (q0 + qb * 32 < N) {
                tma_reduce_add_3d(&tm_dqacc, stg + (qb * 4 + db) * 4096, db * 32, q0 + qb * 32,
                                  w.bh);
                tma_reduce_add_3d(&tm_dqacc, stg + (qb * 4 + db + 1) * 4096, (db + 1) * 32,
                                  q0 + qb * 32, w.bh);
              }
              bulk_commit_group();
              bulk_wait_group_read1();
            }
          }
          bulk_wait_group_read0();
          mbar_arrive(bar(kBStageEmpty + s));
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  } else if (warp >= kParkWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kParkRegs));
    // ================================================================ dQ parking
    // TMEM lanes 32*w4 .. +31 of the dQ columns: query rows 32*(w4 & 1) + lane
    // of this CTA's 64, d columns 64*(w4 >> 1) .. +63 -> boxes (query block
    // w4 & 1, d blocks 2*(w4 >> 1) and +1) of the stage.
    const int w4 = warp & 3;
    const int qb = w4 & 1;
    const int dh = w4 >> 1;
    const uint32_t tQ = tmem + (static_cast<uint32_t>(w4 * 32) << 16) + kColB;
    bool ok = misc[1] == 0u;
    uint32_t step = 0;
    BwdItem w;
    for (int m = 0; ok && get_item2<CAUSAL>(m, n_tiles, args, w); ++m) {
      for (int it = 0; it < w.n_it; ++it, ++step) {
        ok = __all_sync(0xffffffffu, mbar_wait_cl(bar(kBDqFull), step & 1, wc, kWaitDqFull));
        if (!ok) break;
        tc_fence_after();
        const uint32_t stg = sbase + kStageOff + (step & 1) * kStageBytes;
        uint32_t d0[32], d1[32];
        tmem_ld32(tQ, d0);
        tmem_ld32(tQ + 32, d1);
        tmem_ld_wait32(d0);
        reg_fence32(d1);
        // The dQ columns are free for the next dP^T as soon as they are in
        // registers; the stores below only feed the reduce warp.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBDqRead + dq_slot(step)));
        const uint32_t box0 = stg + (qb * 4 + 2 * dh) * 4096 + lane * 128;
        dcheck(in_range(box0, 4096 + 128, stg, stg + kStageBytes), args.status, 505);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const uint32_t sw = static_cast<uint32_t>(c4 ^ (lane & 7)) << 4;
          st_shared_v4(box0 + sw, d0[4 * c4], d0[4 * c4 + 1], d0[4 * c4 + 2], d0[4 * c4 + 3]);
          st_shared_v4(box0 + 4096 + sw, d1[4 * c4], d1[4 * c4 + 1], d1[4 * c4 + 2],
                       d1[4 * c4 + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBDqParked + dq_slot(step)));
      }
    }
  } else if (warp == kRelayWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ relay (rank 1)
    // Each phase of this CTA's warps that the leader's MMAs depend on is
    // passed on with one arrival on the leader's barrier, in the order the
    // leader consumes them.  The data each phase announces is complete when
    // the phase completes (TMEM stores waited for, st.async bytes counted),
    // so the arrival needs no release.
    if (rank == 1) {
      bool ok = misc[1] == 0u;
      uint32_t step = 0;
      BwdItem w;
      auto relay = [&](int local, uint32_t parity, int remote) {
        if (!mbar_wait_cl_warp(bar(local), parity, wc, kWaitPFull)) return false;
        if (local == kBDsqFull) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(lead(remote));
        return true;
      };
      for (int m = 0; ok && get_item2<CAUSAL>(m, n_tiles, args, w); ++m) {
        for (int it = 0; ok && it < w.n_it; ++it, ++step) {
          ok = relay(kBPLocal, step & 1, kBPRemote) && relay(kBDsLocal, step & 1, kBDsRemote) &&
               relay(kBDsqFull, step & 1, kBDsqRemote) &&
               relay(kBDqRead + dq_slot(step), (step >> 1) & 1, kBDqRemote + dq_slot(step));
        }
        if (ok) ok = relay(kBEpiDone, m & 1, kBDkvRemote);
      }
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
  }

  tc_fence_before();
  __syncthreads();
  // The peer may still read this CTA's TMEM and shared memory (its MMAs,
  // remote stores and arrivals) until it, too, is done.
  cluster_sync_all();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

template <bool CAUSAL>
cudaError_t launch_bwd2_t(const CUtensorMap& tq, const CUtensorMap& tq64, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo,
                          const CUtensorMap& tdo64, const CUtensorMap& tacc, const BwdArgs& a,
                          cudaStream_t stream) {
  auto kern = bwd2_kernel<CAUSAL>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  int dev = 0, l2 = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return e;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const long long units = static_cast<long long>((n_tiles + 1) / 2) * a.BH;
  if (units >= 0x3fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // Persistent grid: as many pairs as can be resident at once (at most one
  // per work unit).
  int max_clusters = 0;
  cfg.gridDim = dim3(2);
  if ((e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg)) != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  const int clusters = static_cast<int>(units < max_clusters ? units : max_clusters);
  cfg.gridDim = dim3(2 * clusters);
  BwdArgs ab = a;
  ab.dq_order = nullptr;
  plan_bwd2_schedule(ab, n_tiles, CAUSAL, clusters, l2);
  e = cudaLaunchKernelEx(&cfg, kern, tq, tq64, tk, tv, tdo, tdo64, tacc, ab);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return e;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd2_main(bool causal, const CUtensorMap& tq, const CUtensorMap& tq64,
                             const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                             const CUtensorMap& tdo64, const CUtensorMap& tacc, const BwdArgs& a,
                             cudaStream_t stream) {
  return causal ? launch_bwd2_t<true>(tq, tq64, tk, tv, tdo, tdo64, tacc, a, stream)
                : launch_bwd2_t<false>(tq, tq64, tk, tv, tdo, tdo64, tacc, a, stream);
}

}  // namespace fattn
