// Static work schedule of the persistent backward kernel: which work items
// (K/V tile j of head bh) every CTA processes, and in which order.
//
// The same function runs in the kernel (device) and on the host, where the
// launcher plans the balancing tail and fattn_bwd_schedule reports the
// schedule to callers and tests without a GPU.
#pragma once

#include "fattn_internal.h"

namespace fattn {

// A work item: K/V tile j of head bh, walking n_it Q tiles.  Step it visits
// Q tile i0 + it (causal: i0 = j), or, without a mask and without the ordered
// dQ reduction, (rot + it) mod n_tiles with rot = j, so that the K/V tiles of
// one head start on different Q tiles instead of all reduce-adding into
// tile 0.
struct BwdItem {
  int j, bh, i0, n_it, rot;
};

// The m-th work item of CTA c of a grid of G CTAs (false past its last one).
//
// Items are numbered in sections of sec_heads heads (sized so that a
// section's dQ accumulator, Q, dO, L and D stay in L2 while its items run;
// one section of all heads in the ordered mode and for causal runs that
// cannot be paired) and, inside a section, heaviest first: by j (causal: K/V
// tile j has n_tiles - j Q tiles), heads inner.  They are dealt in snake
// order over the CTAs ("FlashAttention v1～v4" v4 §4: persistent scheduling,
// heaviest first, L2-aware head order).
//
// Causal with paired items (a.paired: even n_tiles, any-order dQ): the CTA's
// items 2q and 2q + 1 are K/V tiles p and n_tiles - 1 - p of one head, the
// q-th pair dealt to it, so every pair walks n_tiles + 1 Q tiles and the
// pairs can be numbered in head sections without unbalancing the CTAs.  The
// pairs cover the first BH - tail_heads heads.  The K/V tiles of the last
// tail_heads heads follow one by one, from the launcher's tables: CTA c
// takes entries tail_off[c] .. tail_off[c + 1] - 1 of tail_item, each
// r * n_tiles + j for K/V tile j of head BH - tail_heads + r.  Whole pairs
// alone would leave the CTAs that get one pair more about n_tiles Q tiles
// behind the others; the single tiles fill that gap.
template <bool CAUSAL>
__host__ __device__ __forceinline__ bool bwd_item(int m, int n_tiles, const BwdArgs& a, int G,
                                                  int c, BwdItem& w) {
  if (CAUSAL && a.paired) {
    const int n_pairs = n_tiles >> 1;
    const int bh_pairs = a.BH - a.tail_heads;
    const int n_paired = n_pairs * bh_pairs;  // < 2^31: the launcher checks n_tiles * BH
    const int rounds = n_paired / G;
    const int pos = (rounds & 1) ? (G - 1 - c) : c;
    const int mine = 2 * (rounds + (pos < n_paired - rounds * G ? 1 : 0));
    if (m < mine) {
      const int q = m >> 1;
      const int kk = q * G + ((q & 1) ? (G - 1 - c) : c);
      const int sec_items = a.sec_heads * n_pairs;
      const int sec = kk / sec_items;
      const int kp = kk - sec * sec_items;
      const int h0 = sec * a.sec_heads;
      const int hs = a.sec_heads < bh_pairs - h0 ? a.sec_heads : bh_pairs - h0;
      const int p = kp / hs;
      w.bh = h0 + kp % hs;
      w.j = (m & 1) ? n_tiles - 1 - p : p;
    } else {
      if (a.tail_heads == 0) return false;
      const int idx = a.tail_off[c] + (m - mine);
      if (idx >= a.tail_off[c + 1]) return false;
      const int e = a.tail_item[idx];
      const int r = e / n_tiles;
      w.bh = bh_pairs + r;
      w.j = e - r * n_tiles;
    }
    w.i0 = w.j;
    w.n_it = n_tiles - w.i0;
    w.rot = 0;
    return true;
  }
  const long long k = static_cast<long long>(m) * G + ((m & 1) ? (G - 1 - c) : c);
  if (k >= static_cast<long long>(n_tiles) * a.BH) return false;
  const int kk = static_cast<int>(k);
  const int sec_items = a.sec_heads * n_tiles;
  const int sec = kk / sec_items;
  const int kp = kk - sec * sec_items;
  const int h0 = sec * a.sec_heads;
  const int hs = a.sec_heads < a.BH - h0 ? a.sec_heads : a.BH - h0;
  w.j = kp / hs;
  w.bh = h0 + kp % hs;
  w.i0 = CAUSAL ? w.j : 0;
  w.n_it = n_tiles - w.i0;
  w.rot = (!CAUSAL && a.dq_order == nullptr) ? w.j : 0;
  return true;
}

// The m-th work item of cluster c of the CTA-pair backward (fattn_bwd2.cu),
// a grid of G clusters of two CTAs.  A work item is a unit u of head bh:
// K/V tiles 2u (cluster rank 0) and 2u + 1 (rank 1), n_units =
// ceil(n_tiles / 2) per head; w.j = 2u.  Causal: the unit walks Q tiles
// 2u .. n_tiles - 1 (rank 1's tile sees a fully masked first Q tile).
// Numbering and dealing follow bwd_item with units in place of K/V tiles:
// head sections, heaviest first, snake order over clusters; causal with an
// even n_units (a.paired): units u and n_units - 1 - u as consecutive items
// (each such pair walks 2 n_tiles - 2 n_units + 2 Q tiles), and the last
// tail_heads heads unit by unit from the launcher's tables (r * n_units + u).
template <bool CAUSAL>
__host__ __device__ __forceinline__ bool bwd2_item(int m, int n_tiles, const BwdArgs& a, int G,
                                                   int c, BwdItem& w) {
  const int n_units = (n_tiles + 1) >> 1;
  int u = 0;
  if (CAUSAL && a.paired) {
    const int n_pairs = n_units >> 1;
    const int bh_pairs = a.BH - a.tail_heads;
    const int n_paired = n_pairs * bh_pairs;
    const int rounds = n_paired / G;
    const int pos = (rounds & 1) ? (G - 1 - c) : c;
    const int mine = 2 * (rounds + (pos < n_paired - rounds * G ? 1 : 0));
    if (m < mine) {
      const int q = m >> 1;
      const int kk = q * G + ((q & 1) ? (G - 1 - c) : c);
      const int sec_items = a.sec_heads * n_pairs;
      const int sec = kk / sec_items;
      const int kp = kk - sec * sec_items;
      const int h0 = sec * a.sec_heads;
      const int hs = a.sec_heads < bh_pairs - h0 ? a.sec_heads : bh_pairs - h0;
      const int p = kp / hs;
      w.bh = h0 + kp % hs;
      u = (m & 1) ? n_units - 1 - p : p;
    } else {
      if (a.tail_heads == 0) return false;
      const int idx = a.tail_off[c] + (m - mine);
      if (idx >= a.tail_off[c + 1]) return false;
      const int e = a.tail_item[idx];
      const int r = e / n_units;
      w.bh = bh_pairs + r;
      u = e - r * n_units;
    }
  } else {
    const long long k = static_cast<long long>(m) * G + ((m & 1) ? (G - 1 - c) : c);
    if (k >= static_cast<long long>(n_units) * a.BH) return false;
    const int kk = static_cast<int>(k);
    const int sec_items = a.sec_heads * n_units;
    const int sec = kk / sec_items;
    const int kp = kk - sec * sec_items;
    const int h0 = sec * a.sec_heads;
    const int hs = a.sec_heads < a.BH - h0 ? a.sec_heads : a.BH - h0;
    u = kp / hs;
    w.bh = h0 + kp % hs;
  }
  w.j = 2 * u;
  w.i0 = CAUSAL ? w.j : 0;
  w.n_it = n_tiles - w.i0;
  w.rot = CAUSAL ? 0 : w.j;
  return true;
}

// Fills the schedule fields of `a` (sec_heads, paired, tail_heads and the
// tail tables) for a launch of `grid` CTAs over n_tiles K/V tiles of a.BH
// heads with head dimension hd, on a device with l2_bytes of L2; `ordered`
// is the deterministic dQ mode.  Requires n_tiles * a.BH < 2^31.
void plan_bwd_schedule(BwdArgs& a, int n_tiles, int hd, bool causal, bool ordered, int grid,
                       long long l2_bytes);

// The same for the CTA-pair backward (bwd2_item): `clusters` pairs of CTAs,
// d = 128, any-order dQ.
void plan_bwd2_schedule(BwdArgs& a, int n_tiles, bool causal, int clusters, long long l2_bytes);

}  // namespace fattn
