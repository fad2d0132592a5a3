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
// and O/l, L are written once at the end.  The row max of an unmasked tile
// comes with S out of TMEM: the .red form of tcgen05.ld (sm_103a) returns each
// thread's maximum of the 32 columns it loads, which removes the 3-input max
// tree from the softmax (measured on GB300, outputs bit-identical: B = 2,
// H = 32, N = 4096 causal with outlier rows 207.3 -> 200.7 us, FP8 182.7 ->
// 176.2 us, d = 64 N = 4096 305.8 -> 297.1 us).
//
// Persistent: one CTA per SM walks work items, each a pair of Q tiles (rows
// [256*pair, 256*pair + 256)) of one (batch, head); with the causal mask
// tile 0 is the upper half (see q_row0).  Items are numbered
// heaviest first (causal: the pairs with the most key tiles) and dealt to the
// CTAs in snake order, so that every CTA gets a similar total; the next item's
// Q load and first S MMAs overlap the current item's last steps and
// epilogue.  Without the mask each slot's Q buffer has its own full / empty
// barrier pair and is refilled as soon as its tile has had its last S, in
// the order Q(tile 0), K_0, Q(tile 1), V_0, ... (measured on GB300 against
// one pair for both buffers, outputs bit-identical: B = 8, H = 16, N = 4096
// 701-708 -> 676-683 us, d = 64 N = 4096 297 -> 293 us; the FP8 forward
// on B = 2, H = 32, N = 4096 causal 174.8-176.2 -> 172.6-172.8 us); the
// causal bf16 items keep one pair for both (see the loader).
//   warps 0-3  softmax of slot 0 (TMEM lanes 0..127, one row per thread)
//   warps 4-7  softmax of slot 1
// A slot is a Q buffer, its TMEM columns and barriers, and the warpgroup
// that serves them; tile t of item m sits in slot slot_of(m, t).
//   warp 8     TMEM allocation + MMA issue (converged warp, elected lane)
//   warp 9     TMA producer (converged warp, elected lane)
//   warps 10-11 idle
// TMEM (512 columns), by slot: S0 [0,128) S1 [128,256) O0 [256,256+d)
// O1 [256+d,256+2d); P (bf16 pairs, 64 columns) aliases the slot's S at
// d = 128 and sits in [384+64s, 448+64s) at d = 64.  Where P aliases S, the
// next S of a slot is issued after its P V; at d = 64 it is issued as soon
// as the softmax has the current S in registers (s_read), and the softmax
// waits for the previous P V (pv_done) before it rescales O or overwrites P
// (measured on GB300: B = 4, H = 16, N = 4096, d = 64 forward 328.2 ->
// 311.9 us).
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

// FP8: Q, K and the transposed V are e4m3 (one byte per element; d = 128
// only), so a row of a tile is one 128-byte swizzle chunk and the ring holds
// twice as many stages.
template <int HD, bool FP8>
struct FwdCfg {
  static_assert(!FP8 || HD == 128, "the FP8 path is built for d = 128");
  static constexpr int kElem = FP8 ? 1 : 2;             // bytes per element
  static constexpr int kRowBytes = HD * kElem;
  static constexpr int kChunks = kRowBytes / 128;       // 128-byte swizzle chunks per row
  static constexpr int kChunkElems = 128 / kElem;
  static constexpr int kChunkBytes = kBM * 128;         // one chunk of a 128-row tile
  static constexpr int kTileBytes = kBM * kRowBytes;
  static constexpr int kKSteps = kRowBytes / 32;        // 32-byte K steps of Q K^T
#ifdef FATTN_FWD_STAGES
  // Test builds: a shallower K/V ring, so that its phases wrap more often.
  // Two stages is the least that works: the MMA order per key tile needs
  // K_{j+1} while V_j is still held.
  static constexpr int kStages = FATTN_FWD_STAGES;
  static_assert(kStages >= 2, "the K/V ring needs two stages");
#else
  static constexpr int kStages = FP8 ? 8 : (HD == 128 ? 4 : 8);
#endif
  static constexpr int kQOff = 0;
  static constexpr int kKvOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKvOff + kStages * kTileBytes;
  // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2],
  // o_empty[2], mma_done, s_read[2], pv_done[2], and slot 1's own q_full /
  // q_empty (unmasked items; causal items share the first pair)
  static constexpr int kNumBars = 2 + 2 * kStages + 8 + 1 + 4 + 2;
  // P has columns of its own (d = 64): the next S can be computed while the
  // softmax still works on the current one.
  static constexpr bool kEarlyS = !FP8 && HD == 64;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
  __device__ static constexpr uint32_t col_s(int t) { return 128u * t; }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + HD * t; }
  __device__ static constexpr uint32_t col_p(int t) {
    return (FP8 || HD == 128) ? 128u * t : 384u + 64u * t;
  }
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct FwdBars {
  uint32_t q_full, q_empty, kv_full0, kv_empty0, s_full[2], p_full[2], o_full[2], o_empty[2],
      mma_done;
};

// A work item: the Q-tile pair starting at row q0 of head bh; tile t sees
// n[t] key tiles (0 when it starts past N), nt = max(n[0], n[1]).
struct Item {
  int q0, bh, n[2], nt;
};

// First query row of tile t of an item.  With the causal mask the upper Q
// tile of the pair has one key tile more and finishes last; it is tile 0,
// whose MMAs each key-tile step issues first, so that at an item boundary
// the next S of the tile that sets the pace is issued first (measured on
// GB300: 1.3 % faster on B = 2, H = 32, N = 4096, 3.4 % at N = 2048).
template <bool CAUSAL>
__device__ __forceinline__ int q_row0(const Item& w, int t) {
  return w.q0 + (CAUSAL ? 1 - t : t) * kBM;
}

template <int V>
struct IntC {
  static constexpr int value = V;
};

// Slot (TMEM columns, Q buffer, barriers, softmax warpgroup) of tile t in
// item m.  With the causal mask the upper tile, which has one key tile more,
// alternates between the two slots: the warpgroup whose lower tile finished
// a key tile earlier takes the next item's upper tile while the other one
// writes its epilogue (measured on GB300: 195.7-196.4 -> 193.4-193.7 us on
// B = 2, H = 32, N = 4096; unmasked runs keep t = slot).
template <bool CAUSAL>
__device__ __forceinline__ int slot_of(int m, int t) {
  return CAUSAL ? (t ^ (m & 1)) : t;
}

// The m-th work item of this CTA: items are numbered in sections of
// sec_heads heads (sized so that a section's K and V stay in L2 while its
// items run) and, inside a section, heaviest first (causal: the Q-tile pairs
// with the most key tiles), heads inner; they are dealt in snake order (round
// m goes left to right when m is even, right to left when odd).  Returns
// false past the last item.
template <bool CAUSAL>
__device__ __forceinline__ bool get_item(int m, int N, int BH, int sec_heads, Item& w) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int num_pairs = (N + 2 * kBM - 1) / (2 * kBM);
  const long long k = static_cast<long long>(m) * G + ((m & 1) ? (G - 1 - c) : c);
  if (k >= static_cast<long long>(num_pairs) * BH) return false;
  // item counts fit in int (the launcher checks num_pairs * BH < 2^31)
  const int kk = static_cast<int>(k);
  const int sec_items = sec_heads * num_pairs;
  const int sec = kk / sec_items;
  const int kp = kk - sec * sec_items;
  const int h0 = sec * sec_heads;
  const int hs = min(sec_heads, BH - h0);
  w.bh = h0 + kp % hs;
  w.q0 = (num_pairs - 1 - kp / hs) * 2 * kBM;
  const int n_kv = (N + kBN - 1) / kBN;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qs = q_row0<CAUSAL>(w, t);
    w.n[t] = qs >= N ? 0 : (CAUSAL ? min(n_kv, qs / kBN + 1) : n_kv);
  }
  w.nt = max(w.n[0], w.n[1]);
  return true;
}

template <int HD, bool CAUSAL, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  using C = FwdCfg<HD, FP8>;
  // Causal bf16 items share one Q barrier pair between the two buffers;
  // unmasked and FP8 items refill each buffer as soon as its tile is done.
  constexpr bool kSharedQ = CAUSAL && !FP8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kBarOff;
  FwdBars b;
  b.q_full = bar0;
  b.q_empty = bar0 + 8;
  b.kv_full0 = bar0 + 16;
  b.kv_empty0 = bar0 + 16 + 8 * C::kStages;
  const uint32_t rest = bar0 + 16 + 16 * C::kStages;
  for (int t = 0; t < 2; ++t) {
    b.s_full[t] = rest + 8 * t;
    b.p_full[t] = rest + 16 + 8 * t;
    b.o_full[t] = rest + 32 + 8 * t;
    b.o_empty[t] = rest + 48 + 8 * t;
  }
  b.mma_done = rest + 64;
  // kEarlyS only: S read into registers / P V complete, per slot.
  auto s_read_bar = [&](int t) { return rest + 72u + 8u * t; };
  auto pv_done_bar = [&](int t) { return rest + 88u + 8u * t; };
  // Q tile of slot s landed / free again: one pair per slot for unmasked
  // items; causal items use b.q_full / b.q_empty for both slots.
  auto q_full_bar = [&](int sl) { return sl ? rest + 104u : b.q_full; };
  auto q_empty_bar = [&](int sl) { return sl ? rest + 112u : b.q_empty; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = args.N;
  const int BH = args.BH;

  if (threadIdx.x == 0) {
    mbar_init(b.q_full, 1);
    mbar_init(b.q_empty, 1);
    mbar_init(rest + 104u, 1);
    mbar_init(rest + 112u, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(b.kv_full0 + 8 * s, 1);
      mbar_init(b.kv_empty0 + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(b.s_full[t], 1);
      mbar_init(b.p_full[t], 4 * 32);
      mbar_init(b.o_full[t], 1);
      mbar_init(b.o_empty[t], 4 * 32);
      if constexpr (C::kEarlyS) {
        mbar_init(s_read_bar(t), 4);
        mbar_init(pv_done_bar(t), 1);
      }
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const WaitCtx wc{args.wait_budget, reinterpret_cast<volatile uint32_t*>(&misc[1]), args.status};

  if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ================================================================ softmax
    const int sl = warp >> 2;             // this warpgroup's slot
    const int wq = warp & 3;
    const int r_tile = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(sl);
    const uint32_t tP = tmem + lane_off + C::col_p(sl);
    const uint32_t tO = tmem + lane_off + C::col_o(sl);
    dcheck(C::col_s(sl) + kBN <= 512 && C::col_o(sl) + HD <= 512 && C::col_p(sl) + 64 <= 512 &&
               ((tmem >> 16) & 0xFFFFu) == 0u,
           args.status, 301);
    float c = args.scale_log2;   // FP8: times the Q and K block scales, per tile pair
    const float tau = args.tau_log2;
    const int n_kv = (N + kBN - 1) / kBN;
    uint32_t s_count = 0;   // S_t tiles consumed so far (phase of s_full / p_full)
    uint32_t o_count = 0;   // items of this tile finished so far (phase of o_full / o_empty)
    bool ok = true;
    Item w;
    for (int m = 0; ok && get_item<CAUSAL>(m, N, BH, args.sec_heads, w); ++m) {
      const int t = slot_of<CAUSAL>(m, sl);   // the item's tile in this slot (involution)
      const int nj = w.n[t];
      if (nj == 0) continue;
      const int qs = q_row0<CAUSAL>(w, t);
      const int row = qs + r_tile;
      float m_ref = -INFINITY;  // running reference max, log2 units
      float l = 0.f;            // sum of the fp32 probabilities (gives L)
      // Sum, over the tiles, of the bf16 rounding error of the probability
      // of each tile's largest score.  P V uses bf16 probabilities while l
      // sums fp32 ones; for a row dominated by one key that mismatch alone
      // would leave O off by up to 2^-9 |v|, so O is normalised by l + l_fix,
      // which is exact for the dominating key.  (The other keys' rounding
      // errors stay, each weighted by its own small share of the row.)
      float l_fix = 0.f;
      // FP8 ("FlashAttention v1～v4" v3 §3, block quantization): S = sq_i sk_j
      // (Q8 K8^T), so the exponent multiplier is scale*log2e*sq_i*sk_j; V_j =
      // sv_j V8_j is folded into the probabilities as rho_j = sv_j / sv_max
      // (<= 1, so P rho stays within e4m3 range) and O is multiplied by
      // sv_max once at the end.
      float c_q = 0.f, sv_max = 1.f;
      if constexpr (FP8) {
        const float* svh = args.sv + static_cast<size_t>(w.bh) * n_kv;
        sv_max = 0.f;
        for (int jj = 0; jj < n_kv; ++jj) sv_max = fmaxf(sv_max, __ldg(svh + jj));
        c_q = args.scale_log2 * __ldg(args.sq + static_cast<size_t>(w.bh) * n_kv + qs / kBM);
      }
      for (int j = 0; j < nj; ++j) {
        // FP8: rho_j enters the exponent as log2(rho_j) (one FMA gives P rho),
        // and the row sum is taken of P rho and multiplied by 1/rho_j.  The
        // offset is clamped at -100: probabilities scaled further down round
        // to e4m3 zero either way, and the sum stays finite.
        float lrho = 0.f, inv_rho = 1.f;
        if constexpr (FP8) {
          c = c_q * __ldg(args.sk + static_cast<size_t>(w.bh) * n_kv + j);
          const float rho = __ldg(args.sv + static_cast<size_t>(w.bh) * n_kv + j) / sv_max;
          lrho = fmaxf(__log2f(rho), -100.f);
          inv_rho = ex2_approx(-lrho);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(b.s_full[sl], s_count & 1, wc, kWaitSFull));
        if (!ok) break;
        ++s_count;
        tc_fence_after();
        // S with each 32-column group's maximum from the TMEM loads themselves
        uint32_t s0[32], s1[32], s2[32], s3[32];
        float mg[4];
        tmem_ld32_max(tS + 0, s0, mg[0]);
        tmem_ld32_max(tS + 32, s1, mg[1]);
        tmem_ld32_max(tS + 64, s2, mg[2]);
        tmem_ld32_max(tS + 96, s3, mg[3]);
        tmem_ld_wait32(s0);
        reg_fence32(s1);
        reg_fence32(s2);
        reg_fence32(s3);
#pragma unroll
        for (int g = 0; g < 4; ++g) reg_fence1(mg[g]);
        // The previous P V of this slot (it reads P and accumulates into O)
        // must have completed before O is rescaled or P overwritten.  With
        // the early next S (kEarlyS) the completion of S no longer implies
        // it, so it is waited for once per step, when first needed.
        bool pv_waited = s_count < 2;
        if constexpr (C::kEarlyS) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_read_bar(sl));
        }
        uint32_t* sv[4] = {s0, s1, s2, s3};
        const int kv0 = j * kBN;
        const bool need_mask = (kv0 + kBN > N) || (CAUSAL && kv0 + kBN - 1 > qs);
        if (need_mask) {
          // columns kv0 + c with c < lim are visible: c < N - kv0 and, causal,
          // kv0 + c <= row
          const int lim = (CAUSAL ? min(N, row + 1) : N) - kv0;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (g * 32 + i >= lim) sv[g][i] = __float_as_uint(-INFINITY);
          }
          // The loads' maxima include the masked columns: the row max of
          // this tile is taken again, as four independent 3-input max chains.
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
        }
        const float mx = fmaxf(fmax3(mg[0], mg[1], mg[2]), mg[3]);
        const float m_new = mx * c;
        const bool need = m_new > m_ref + tau;
        // O must be rescaled by alpha = 2^(m_old - m_new) before P V_j is
        // added; that is done below, once S is out of the registers, so that
        // all of O can be in flight at once.
        const bool rescale = __any_sync(0xffffffffu, need);
        float alpha = 1.f;
        if (rescale) {
          alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
          if (need) m_ref = m_new;
          l *= alpha;
          l_fix *= alpha;
        }
        // exponent offset of the element loop: -m_ref, and log2(rho_j) for FP8
        const float nm = FP8 ? -m_ref + lrho : -m_ref;
        {
          // the same arithmetic as the element loop below, for the largest score
          const float p_top = ex2_approx(fmaf(mx, c, -m_ref));
          if constexpr (FP8)
            l_fix += round_e4m3(ex2_approx(fmaf(mx, c, nm))) * inv_rho - p_top;
          else
            l_fix += __bfloat162float(__float2bfloat16_rn(p_top)) - p_top;
        }
        const uint64_t c2 = splat2(c);
        const uint64_t nm2 = splat2(nm);
        // Two columns per instruction (packed fp32 pairs); partial sums per
        // 32-column group keep the additions independent.
        if constexpr (C::kEarlyS) {
          if (!pv_waited) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(pv_done_bar(sl), (s_count - 2) & 1, wc, kWaitPFull));
            pv_waited = true;
            if (!ok) break;
            tc_fence_after();
          }
        }
        uint64_t rs2[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t pk[16];
          uint64_t e2 = 0ull;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            uint32_t x0, x1;
            unpack2(ffma2(pack2(sv[g][2 * i], sv[g][2 * i + 1]), c2, nm2), x0, x1);
            const float a0 = ex2_approx(__uint_as_float(x0));
            const float a1 = ex2_approx(__uint_as_float(x1));
            if constexpr (FP8) {   // P rho, kept in the score registers until packed
              sv[g][2 * i] = __float_as_uint(a0);
              sv[g][2 * i + 1] = __float_as_uint(a1);
            } else {
              pk[i] = pack_bf16x2(a0, a1);
            }
            e2 = fadd2(e2, pack2(__float_as_uint(a0), __float_as_uint(a1)));
          }
          if constexpr (FP8) {
            // e4m3, four per TMEM column (K order), 8 columns per 32 keys
#pragma unroll
            for (int q = 0; q < 8; ++q)
              pk[q] = pack_e4m3x4(__uint_as_float(sv[g][4 * q]), __uint_as_float(sv[g][4 * q + 1]),
                                  __uint_as_float(sv[g][4 * q + 2]),
                                  __uint_as_float(sv[g][4 * q + 3]));
            tmem_st8(tP + 8 * g, pk);
          } else {
            tmem_st16(tP + 16 * g, pk);
          }
          rs2[g] = e2;
        }
        if (rescale && j > 0) {
          // P V_{j-1} has completed: it was issued before S_j, whose
          // completion was waited for (d = 64: waited for above).  All of
          // O in flight at once: measured on GB300, forward 217.7 -> 210.6 us
          // on the B = 2, H = 32, N = 4096 causal workload with its x20
          // outlier rows (about half of its steps rescale), FP8 195 -> 181 us,
          // unmasked shapes unchanged, causal N = 16384 without outliers
          // 2 % slower.
          if constexpr (C::kEarlyS) {
            if (!pv_waited) {
              ok = __all_sync(0xffffffffu,
                              mbar_wait(pv_done_bar(sl), (s_count - 2) & 1, wc, kWaitPFull));
              pv_waited = true;
              if (!ok) break;
              tc_fence_after();
            }
          }
          uint32_t o[HD / 32][32];
#pragma unroll
          for (int ch = 0; ch < HD / 32; ++ch) tmem_ld32(tO + 32 * ch, o[ch]);
          tmem_ld_wait32(o[0]);
#pragma unroll
          for (int ch = 1; ch < HD / 32; ++ch) reg_fence32(o[ch]);
          const uint64_t a2 = splat2(alpha);
#pragma unroll
          for (int ch = 0; ch < HD / 32; ++ch) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              unpack2(fmul2(pack2(o[ch][2 * i], o[ch][2 * i + 1]), a2), o[ch][2 * i],
                      o[ch][2 * i + 1]);
            tmem_st32(tO + 32 * ch, o[ch]);
          }
        }
        float rs[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t u0, u1;
          unpack2(rs2[g], u0, u1);
          rs[g] = __uint_as_float(u0) + __uint_as_float(u1);
        }
        if constexpr (FP8)
          l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) * inv_rho;
        else
          l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b.p_full[sl]);
      }
      if (!ok) break;
      // ---- epilogue: O / l_bf -> bf16 to global, L = (m + log2 l) ln 2.  O_t
      // is read out of TMEM whole (each thread its own row) and handed back
      // to the MMA warp before the stores.
      ok = __all_sync(0xffffffffu, mbar_wait(b.o_full[sl], o_count & 1, wc, kWaitOFull));
      if (!ok) break;
      ++o_count;
      tc_fence_after();
      const float inv = sv_max / (l + l_fix);   // sv_max = 1 unless FP8
      const bool row_ok = row < N;
      uint32_t pw[HD / 2];   // the row as bf16 pairs; 16-byte chunk c = words 4c .. 4c + 3
#pragma unroll
      for (int ch = 0; ch < HD / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(tO + 32 * ch, o);
        tmem_ld_wait32(o);
        const uint64_t i2 = splat2(inv);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t y0, y1;
          unpack2(fmul2(pack2(o[2 * i], o[2 * i + 1]), i2), y0, y1);
          pw[16 * ch + i] = pack_bf16x2(__uint_as_float(y0), __uint_as_float(y1));
        }
      }
      tc_fence_before();
      mbar_arrive(b.o_empty[sl]);
      // Stores of whole 128-byte lines.  Row-per-thread stores would put 32
      // lines into every warp store, 16 bytes each, and the L1 traffic they
      // cause slows the MMAs' shared-memory operand reads (measured on GB300:
      // 5-10 % of the kernel).  So the 8 lanes of each group first exchange
      // 16-byte chunks, an 8 x 8 transpose per 128-byte half row in three
      // XOR-shuffle stages: afterwards lane i of group g holds, in chunk slot
      // 8h + j, chunk 8h + i of the group's row j, and one warp store writes
      // 8 lanes x 16 bytes of one row for each of the four groups.
      const int li = lane & 7;
#pragma unroll
      for (int h = 0; h < HD / 64; ++h) {
#pragma unroll
        for (int dd = 4; dd >= 1; dd >>= 1) {
          const bool up = (li & dd) != 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j & dd) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t lo = pw[4 * (8 * h + j) + q];
              const uint32_t hi = pw[4 * (8 * h + j + dd) + q];
              const uint32_t got = __shfl_xor_sync(0xffffffffu, up ? lo : hi, dd);
              pw[4 * (8 * h + j) + q] = up ? got : lo;
              pw[4 * (8 * h + j + dd) + q] = up ? hi : got;
            }
          }
        }
      }
      const int grow0 = qs + wq * 32 + (lane & ~7);   // the group's row 0
#pragma unroll
      for (int h = 0; h < HD / 64; ++h) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const size_t o_idx = (static_cast<size_t>(w.bh) * N + grow0 + j) * HD + 64 * h + 8 * li;
          if (grow0 + j < N &&
              dcheck(o_idx + 8 <= static_cast<size_t>(BH) * N * HD, args.status, 302)) {
            uint4* dst = reinterpret_cast<uint4*>(args.o + o_idx);
            __stcs(dst, make_uint4(pw[4 * (8 * h + j)], pw[4 * (8 * h + j) + 1],
                                   pw[4 * (8 * h + j) + 2], pw[4 * (8 * h + j) + 3]));
          }
        }
      }
      if (row_ok && dcheck(static_cast<size_t>(w.bh) * N + row < static_cast<size_t>(BH) * N,
                           args.status, 303))
        args.lse[static_cast<size_t>(w.bh) * N + row] = (m_ref + log2f(l)) * kLn2;
    }
  } else if (warp == kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    // ================================================================ MMA issue
    // The whole warp runs this (converged); one elected lane issues.
    {
      constexpr uint32_t idesc_qk =
          FP8 ? idesc_e4m3_f32(kBM, kBN) : idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv =
          FP8 ? idesc_e4m3_f32(kBM, HD) : idesc_bf16_f32(kBM, HD, false, true);
      auto kv_smem = [&](uint32_t i) {
        return sbase + C::kKvOff + (i % C::kStages) * C::kTileBytes;
      };
      auto kv_full = [&](uint32_t i) { return b.kv_full0 + 8u * (i % C::kStages); };
      auto kv_empty = [&](uint32_t i) { return b.kv_empty0 + 8u * (i % C::kStages); };
      auto kv_parity = [&](uint32_t i) { return (i / C::kStages) & 1u; };
      // S_t = Q_t K^T: M = 128, N = 128, K = HD in steps of 32 bytes (16
      // bf16 or 32 e4m3 elements) inside a 128-byte swizzle row, then the
      // next 128-byte chunk.  The descriptors are built once and advanced by
      // constant offsets (their start-address field is in 16-byte units).
      auto issue_s = [&](int t, uint32_t ik) {
        const uint64_t da = sdesc_sw128(sbase + C::kQOff + t * C::kTileBytes, 16, 1024);
        const uint64_t db = sdesc_sw128(kv_smem(ik), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < C::kKSteps; ++kk) {
          const uint32_t off = ((kk >> 2) * C::kChunkBytes + (kk & 3) * 32) >> 4;
          if constexpr (FP8)
            mma_ss_f8_w(tmem + C::col_s(t), da + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
          else
            mma_ss_w(tmem + C::col_s(t), da + off, db + off, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t V: A = P_t from TMEM (8 columns per K step: 16 bf16 or 32
      // e4m3 keys).  bf16: B = the V tile, MN-major (d contiguous): K step =
      // 16 rows = 2048 bytes, the next 64 columns of d one chunk (16 KiB)
      // away.  FP8: B = the transposed V tile (d rows of 128 key bytes),
      // K-major, K step = 32 bytes.
      auto issue_pv = [&](int t, uint32_t iv, uint32_t acc) {
        if constexpr (FP8) {
          const uint64_t dv = sdesc_sw128(kv_smem(iv), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 32; ++kk)
            mma_ts_f8_w(tmem + C::col_o(t), tmem + C::col_p(t) + 8 * kk, dv + ((kk * 32) >> 4),
                        idesc_pv, kk > 0 ? 1u : acc);
        } else {
          const uint64_t dv = sdesc_sw128(kv_smem(iv), C::kChunkBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_w(tmem + C::col_o(t), tmem + C::col_p(t) + 8 * kk, dv + ((kk * 2048) >> 4),
                     idesc_pv, kk > 0 ? 1u : acc);
        }
      };
      uint32_t kvb = 0;                      // ring index of this item's first K tile
      // Per tile of the current item (kept in registers: the slots' counters
      // trade places whenever the slot mapping does).
      uint32_t p_count[2] = {0u, 0u};        // P tiles consumed in the tile's slot (p_full phase)
      uint32_t o_count[2] = {0u, 0u};        // items finished in the tile's slot (o_empty phase)
      uint32_t qm[2] = {0u, 0u};             // unmasked: Q tiles consumed per slot (q_full phase)
      Item w{};
      // One item; F = the slot of the upper tile, a compile-time constant so
      // that every TMEM column and shared-memory address below folds.
      auto run_item = [&](auto f_c, int m) -> bool {
        constexpr int F = decltype(f_c)::value;
        const int nt = w.nt;
        // S(0) may overwrite the slot's S / P: the previous item's P V MMAs
        // that read P there were issued earlier, and MMAs complete in issue
        // order.
        bool k0_ready = false;
        if constexpr (kSharedQ) {   // one Q barrier pair for both buffers (see the loader)
          if (!mbar_wait_warp(b.q_full, m & 1, wc, kWaitQFull)) return false;
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (w.n[t] > 0) {
            const int sl = t ^ F;
            if constexpr (!kSharedQ) {
              if (!mbar_wait_warp(q_full_bar(sl), qm[sl] & 1, wc, kWaitQFull)) return false;
              ++qm[sl];
            }
            if (!k0_ready) {
              if (!mbar_wait_warp(kv_full(kvb), kv_parity(kvb), wc, kWaitKvFull)) return false;
              k0_ready = true;
            }
            tc_fence_after();
            issue_s(sl, kvb);
            mma_commit_w(b.s_full[sl]);
            if (!kSharedQ && w.n[t] == 1) mma_commit_w(q_empty_bar(sl));   // the tile's only S
          }
        }
        mma_commit_w(kv_empty(kvb));
        if (kSharedQ && nt == 1) mma_commit_w(b.q_empty);   // every S MMA of the item is issued
        for (int j = 0; j < nt; ++j) {
          const uint32_t iv = kvb + 2 * j + 1;
          const uint32_t ikn = kvb + 2 * j + 2;
          if (!mbar_wait_warp(kv_full(iv), kv_parity(iv), wc, kWaitKvFull)) return false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int sl = t ^ F;
            if constexpr (C::kEarlyS) {
              if (t == 0 && j + 1 < nt) {
                if (!mbar_wait_warp(kv_full(ikn), kv_parity(ikn), wc, kWaitKvFull)) return false;
              }
              if (j < w.n[t]) {
                // The softmax has S(j) in registers: S(j + 1) may go into its
                // columns while the softmax and P V(j) proceed.
                if (!mbar_wait_warp(s_read_bar(sl), p_count[t] & 1, wc, kWaitPFull)) return false;
                tc_fence_after();
                if (j + 1 < w.n[t]) {
                  issue_s(sl, ikn);
                  mma_commit_w(b.s_full[sl]);
                  if (!kSharedQ && j + 2 == w.n[t]) mma_commit_w(q_empty_bar(sl));   // the tile's last S
                }
              }
            }
            if (j < w.n[t]) {
              if (j == 0 && o_count[t] > 0 &&
                  !mbar_wait_warp(b.o_empty[sl], (o_count[t] - 1) & 1, wc, kWaitOFull))
                return false;   // the slot's previous O has been read out
              if (!mbar_wait_warp(b.p_full[sl], p_count[t] & 1, wc, kWaitPFull)) return false;
              ++p_count[t];
              tc_fence_after();
              issue_pv(sl, iv, j > 0 ? 1u : 0u);
              if constexpr (C::kEarlyS) mma_commit_w(pv_done_bar(sl));
              if (j == w.n[t] - 1) mma_commit_w(b.o_full[sl]);
            }
            if constexpr (!C::kEarlyS) {
              if (t == 0 && j + 1 < nt) {
                if (!mbar_wait_warp(kv_full(ikn), kv_parity(ikn), wc, kWaitKvFull)) return false;
                tc_fence_after();
              }
              if (j + 1 < w.n[t]) {
                issue_s(sl, ikn);
                mma_commit_w(b.s_full[sl]);
                if (!kSharedQ && j + 2 == w.n[t]) mma_commit_w(q_empty_bar(sl));   // the tile's last S
              }
            }
          }
          mma_commit_w(kv_empty(iv));
          if (j + 1 < nt) mma_commit_w(kv_empty(ikn));
          if (kSharedQ && j + 2 == nt) mma_commit_w(b.q_empty);   // the last S MMAs are issued
        }
        return true;
      };
      for (int m = 0; get_item<CAUSAL>(m, N, BH, args.sec_heads, w); ++m) {
        if (CAUSAL && m > 0) {
          // The slot mapping flips every item; the counters follow the slots.
          uint32_t x = p_count[0];
          p_count[0] = p_count[1];
          p_count[1] = x;
          x = o_count[0];
          o_count[0] = o_count[1];
          o_count[1] = x;
        }
        const bool item_ok = (CAUSAL && (m & 1)) ? run_item(IntC<1>{}, m) : run_item(IntC<0>{}, m);
        if (!item_ok) goto mma_end;
        for (int t = 0; t < 2; ++t) o_count[t] += w.n[t] > 0 ? 1u : 0u;
        kvb += 2 * w.nt;
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
      uint32_t kvb = 0;      // ring index of the next K/V load
      uint32_t ql[2] = {0u, 0u};   // unmasked: Q tiles loaded per slot
      int items = 0;               // causal: items whose Q pair was loaded
      // Q is read once; K and V are read again by the other Q-tile pairs of
      // the head: keep them in L2 ahead of Q and O (O is stored with the
      // streaming hint).  Measured on GB300, B = 2, H = 32, N = 4096 causal:
      // DRAM 594 -> 574 MB per launch (FP8 207 -> 172 MB), time unchanged.
      const uint64_t pol_q = l2_evict_first_policy();
      const uint64_t pol_kv = l2_evict_last_policy();
      Item w;
      bool aborted = false;
      for (int m = 0; !aborted && get_item<CAUSAL>(m, N, BH, args.sec_heads, w); ++m) {
        // Unmasked and FP8: Q of tile t into its slot once that slot's
        // previous Q tile has had its last S, in the order Q(tile 0), K_0,
        // Q(tile 1), V_0, ...  Causal bf16: both Q tiles of the item once the
        // previous item's last S MMAs are issued, then K_0 -- inside a
        // forward + backward step the per-slot refill measured ~1 % slower
        // for the causal mask (while faster for forward calls on their own).
        auto load_q = [&](int t) -> bool {
          if (w.n[t] == 0) return true;
          const int sl = slot_of<CAUSAL>(m, t);
          if (ql[sl] > 0 &&
              !mbar_wait_warp(q_empty_bar(sl), (ql[sl] - 1) & 1, wc, kWaitKvEmpty))
            return false;
          mbar_arrive_expect_tx_w(q_full_bar(sl), C::kTileBytes);
          for (int cc = 0; cc < C::kChunks; ++cc)
            tma_load_3d_hint_w(sbase + C::kQOff + sl * C::kTileBytes + cc * C::kChunkBytes, &tm_q,
                               q_full_bar(sl), cc * C::kChunkElems, q_row0<CAUSAL>(w, t), w.bh,
                               pol_q);
          ++ql[sl];
          return true;
        };
        if constexpr (kSharedQ) {
          if (m > 0 && !mbar_wait_warp(b.q_empty, (m - 1) & 1, wc, kWaitKvEmpty)) break;
          uint32_t qbytes = 0;
          for (int t = 0; t < 2; ++t) qbytes += w.n[t] > 0 ? C::kTileBytes : 0;
          mbar_arrive_expect_tx_w(b.q_full, qbytes);
          for (int t = 0; t < 2; ++t) {
            if (w.n[t] == 0) continue;
            for (int cc = 0; cc < C::kChunks; ++cc)
              tma_load_3d_hint_w(sbase + C::kQOff + slot_of<CAUSAL>(m, t) * C::kTileBytes +
                                     cc * C::kChunkBytes,
                                 &tm_q, b.q_full, cc * C::kChunkElems, q_row0<CAUSAL>(w, t),
                                 w.bh, pol_q);
          }
          items = m + 1;
        } else {
          if (!load_q(0)) break;
        }
        for (int i = 0; i < 2 * w.nt; ++i) {
          const uint32_t r = kvb + i;
          const uint32_t s = r % C::kStages;
          const uint32_t rnd = r / C::kStages;
          if (rnd > 0 &&
              !mbar_wait_warp(b.kv_empty0 + 8u * s, (rnd - 1) & 1, wc, kWaitKvEmpty)) {
            aborted = true;
            kvb = r;
            break;
          }
          const uint32_t full = b.kv_full0 + 8u * s;
          mbar_arrive_expect_tx_w(full, C::kTileBytes);
          const CUtensorMap* tm = (i & 1) ? &tm_v : &tm_k;
          const uint32_t dst = sbase + C::kKvOff + s * C::kTileBytes;
          dcheck(in_range(dst, C::kTileBytes, sbase + C::kKvOff, sbase + C::kBarOff), args.status,
                 304);
          if (FP8 && (i & 1)) {
            // transposed V: d rows x 128 key bytes starting at key (i/2)*128
            tma_load_3d_hint_w(dst, tm, full, (i >> 1) * kBN, 0, w.bh, pol_kv);
          } else {
            for (int cc = 0; cc < C::kChunks; ++cc)
              tma_load_3d_hint_w(dst + cc * C::kChunkBytes, tm, full, cc * C::kChunkElems,
                                 (i >> 1) * kBN, w.bh, pol_kv);
          }
          if (!kSharedQ && i == 0 && !load_q(1)) {
            aborted = true;
            kvb = r + 1;
            break;
          }
        }
        if (aborted) break;
        kvb += 2 * w.nt;
      }
      // Every copy this warp started must have landed before the CTA exits.
      for (uint32_t r = kvb > C::kStages ? kvb - C::kStages : 0; r < kvb; ++r)
        mbar_wait_drain(b.kv_full0 + 8u * (r % C::kStages), (r / C::kStages) & 1,
                        args.wait_budget);
      for (int sl = 0; sl < 2; ++sl)
        if (ql[sl] > 0) mbar_wait_drain(q_full_bar(sl), (ql[sl] - 1) & 1, args.wait_budget);
      if (items > 0) mbar_wait_drain(b.q_full, (items - 1) & 1, args.wait_budget);
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

template <int HD, bool CAUSAL, bool FP8>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<HD, FP8>;
  auto kern = fwd_kernel<HD, CAUSAL, FP8>;
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
  const long long items = static_cast<long long>((a.N + 2 * kBM - 1) / (2 * kBM)) * a.BH;
  if (items >= 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(items < sms ? items : sms));
  // Heads per section: a third of L2 over one head's K and V, which every
  // Q-tile pair of the head reads.  Only without a mask: causal items weigh
  // from 2 to N/128 key tiles and are dealt to the CTAs statically, which
  // balances only when the whole order runs heaviest first (sections made
  // the causal forward 19-29 % slower on GB300).
  FwdArgs ab = a;
  ab.sec_heads = a.BH;
  if (!CAUSAL) {
    const long long per_head =
        static_cast<long long>((a.N + kBN - 1) / kBN) * 2 * C::kTileBytes;
    const long long fit = per_head > 0 ? (static_cast<long long>(l2) / 3) / per_head : 1;
    ab.sec_heads = static_cast<int>(fit < 1 ? 1 : (fit > a.BH ? a.BH : fit));
  }
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, ab);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdArgs& a, cudaStream_t stream) {
  if (d == 64) {
    return causal ? launch_fwd_t<64, true, false>(tq, tk, tv, a, stream)
                  : launch_fwd_t<64, false, false>(tq, tk, tv, a, stream);
  }
  return causal ? launch_fwd_t<128, true, false>(tq, tk, tv, a, stream)
                : launch_fwd_t<128, false, false>(tq, tk, tv, a, stream);
}

cudaError_t launch_fwd_fp8(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const FwdArgs& a, cudaStream_t stream) {
  return causal ? launch_fwd_t<128, true, true>(tq, tk, tv, a, stream)
                : launch_fwd_t<128, false, true>(tq, tk, tv, a, stream);
}

}  // namespace fattn
