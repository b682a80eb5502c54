// swa_sched.h — the work-item arithmetic of the band / varlen tile schedule,
// shared by the kernels (device) and the host (launch sizing and the
// schedule export that the host tests check).
//
// The BAND window (FlashAttentionVarLenScore doc, parameters preTokens /
// nextTokens as the left and right edges): query i sees key j iff
// i - pre <= j <= i + next, indices local to the sequence; sparse_mode 0
// sees every key.  A 128-row query tile therefore touches one contiguous run
// of 128-row key tiles and a key tile one contiguous run of query tiles;
// tiles outside those runs are never visited.
#pragma once
#include <cstdint>

#include "swa_internal.h"

#if defined(__CUDACC__)
#define SWA_HD __host__ __device__ __forceinline__
#else
#define SWA_HD inline
#endif

namespace swa {

// A resolved work item: which (batch, head, tile) a CTA owns, and the
// geometry of its sequence.
struct Item {
  int b, n, tile;
  SeqInfo s;
};

// Work item k of a launch's table.  `nh` is the number of heads per batch
// the table enumerates: query heads for the query-major kernels, key/value
// heads for the key-major one.
template <int CAP>
SWA_HD Item resolve_item(const SeqTable<CAP>& tab, const Geometry& g, int k, int nh) {
  int lo = 0, hi = tab.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tab.d[mid].item_begin <= k) lo = mid; else hi = mid - 1;
  }
  const SeqDesc& d = tab.d[lo];
  const int local = k - d.item_begin;
  const int h = local / d.tiles;  // head by head: the CTAs in flight share a head's tiles in L2
  const int rank = local - h * d.tiles;
  Item it;
  it.tile = d.descending ? d.tiles - 1 - rank : rank;
  if (d.b < 0) {
    it.b = h / nh;
    it.n = h - it.b * nh;
    it.s.mask_base = static_cast<int64_t>(it.b) * g.N * g.S_q * static_cast<int64_t>(g.S_kv);
  } else {
    it.b = d.b;
    it.n = h;
    it.s.mask_base = d.mask_base;
  }
  it.s.q_start = d.q_start;
  it.s.q_len = d.q_len;
  it.s.kv_start = d.kv_start;
  it.s.kv_len = d.kv_len;
  return it;
}

// Key tiles [*t0, *t0 + *n) that query tile `tile` of sequence s touches.
SWA_HD void key_tiles_of_query_tile(const Geometry& g, const SeqInfo& s, int tile, int* t0, int* n) {
  const int q0 = tile * kTileM;
  const int q_last = q0 + kTileM - 1 < s.q_len - 1 ? q0 + kTileM - 1 : s.q_len - 1;
  int lo = 0, hi = s.kv_len - 1;
  if (g.sparse_mode == 4) {
    lo = q0 - g.pre > lo ? q0 - g.pre : lo;
    hi = q_last + g.next < hi ? q_last + g.next : hi;
  }
  *t0 = 0;
  *n = 0;
  if (lo <= hi) {
    *t0 = lo / kTileN;
    *n = hi / kTileN - *t0 + 1;
  }
}

// Key tiles [*u0, *u0 + *n) that query tiles 2p and 2p + 1 of sequence s
// visit between them (the forward at D <= 64 takes the two in one CTA; the
// second may not exist).  A tile with no visible key adds nothing; the union
// of two runs is taken from the first start to the last end.
SWA_HD void key_tiles_of_query_pair(const Geometry& g, const SeqInfo& s, int p, int* u0, int* n) {
  int ta = 0, na = 0, tb = 0, nb = 0;
  if (2 * p * kTileM < s.q_len) key_tiles_of_query_tile(g, s, 2 * p, &ta, &na);
  if ((2 * p + 1) * kTileM < s.q_len) key_tiles_of_query_tile(g, s, 2 * p + 1, &tb, &nb);
  *u0 = 0;
  *n = 0;
  if (na > 0 && nb > 0) {
    *u0 = ta < tb ? ta : tb;
    *n = (ta + na > tb + nb ? ta + na : tb + nb) - *u0;
  } else if (na > 0) {
    *u0 = ta;
    *n = na;
  } else if (nb > 0) {
    *u0 = tb;
    *n = nb;
  }
}

// Query tiles [*t0, *t0 + *n) that see key tile `tile` of sequence s:
// i - pre <= j <= i + next  <=>  j - next <= i <= j + pre.
SWA_HD void query_tiles_of_key_tile(const Geometry& g, const SeqInfo& s, int tile, int* t0, int* n) {
  const int j0 = tile * kTileN;
  const int j_last = j0 + kTileN - 1 < s.kv_len - 1 ? j0 + kTileN - 1 : s.kv_len - 1;
  int lo = 0, hi = s.q_len - 1;
  if (g.sparse_mode == 4) {
    lo = j0 - g.next > lo ? j0 - g.next : lo;
    hi = j_last + g.pre < hi ? j_last + g.pre : hi;
  }
  *t0 = 0;
  *n = 0;
  if (lo <= hi) {
    *t0 = lo / kTileM;
    *n = hi / kTileM - *t0 + 1;
  }
}

}  // namespace swa
