// Block-wide top-K selection over order-preserving uint32 keys held in shared memory.
//
// radix_select finds a threshold T and a count `need` such that the top-k keys are exactly the
// keys > T plus the `need` lowest-indexed keys == T.  It resolves 8-bit digits from the highest
// bit where the valid keys differ (the common prefix, found from their min and max, is skipped),
// with per-warp private histograms (no same-address contention across warps), and stops as soon
// as the bin holding the k-th key is taken whole (then T = bin start - 1, need = 0) — for
// continuous scores that is usually after two passes.  compact_ascending writes the selected
// indices in ascending order, so equal keys resolve to the lower index: the tie rule.
#pragma once

#include "common.cuh"

namespace dsa {

struct Selection {
  uint32_t thresh;  // keys > thresh are selected
  int need;         // plus this many keys == thresh, lowest indices first
  int n_valid;      // keys != 0
};

template <int NT>
struct SelectScratch {
  static constexpr int kWarps = NT / 32;
  int hist[kWarps][256];  // per-warp private histograms
  int tot[256];
  int red[33];
  uint32_t kmin[kWarps], kmax[kWarps];
  int digit, above, bin;
  uint32_t lo, hi;
};

template <int NT>
DSA_DEV Selection radix_select(const uint32_t* keys, int n, int k, SelectScratch<NT>& sh) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int c = 0;
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int j = tid; j < n; j += NT) {
    const uint32_t key = keys[j];
    if (key != 0u) {
      ++c;
      mn = min(mn, key);
      mx = max(mx, key);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sh.kmin[warp] = mn;
    sh.kmax[warp] = mx;
  }
  int n_valid;
  block_exclusive_scan(c, sh.red, &n_valid);  // also orders the writes above
  Selection sel;
  sel.n_valid = n_valid;
  if (k >= n_valid) {
    sel.thresh = 0u;
    sel.need = 0;
    return sel;
  }
  if (k <= 0) {
    sel.thresh = 0xffffffffu;
    sel.need = 0;
    return sel;
  }
  mn = 0xffffffffu;
  mx = 0u;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    mn = min(mn, sh.kmin[w]);
    mx = max(mx, sh.kmax[w]);
  }
  const uint32_t diff = mn ^ mx;
  // first digit: the 8-bit group holding the highest differing bit (all keys equal: last group)
  int shift = diff == 0u ? 0 : ((31 - __clz(diff)) / 8) * 8;
  uint32_t prefix = mn & ~((shift >= 24) ? 0xffffffffu : ((1u << (shift + 8)) - 1u));
  uint32_t mask = (shift >= 24) ? 0u : ~((1u << (shift + 8)) - 1u);
  int remaining = k;
  const int iters = (n + NT - 1) / NT;
  for (;; shift -= 8) {
    int* hw = sh.hist[warp];
    for (int e = lane; e < 256; e += 32) hw[e] = 0;
    __syncwarp();
    for (int it = 0; it < iters; ++it) {
      const int j = it * NT + tid;
      const uint32_t key = j < n ? keys[j] : 0u;
      if (key != 0u && (key & mask) == prefix) atomicAdd(&hw[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    for (int e = tid; e < 256; e += NT) {
      int s = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) s += sh.hist[w][e];
      sh.tot[e] = s;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255-8l .. 248-8l (from the top); find the bin where the count of keys
      // at or above it first reaches `remaining`.
      int loc[8], s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        loc[q] = sh.tot[255 - (lane * 8 + q)];
        s += loc[q];
      }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int above = incl - s;
      if (above < remaining && incl >= remaining) {
        int cum = above;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (cum + loc[q] >= remaining) {
            sh.digit = 255 - (lane * 8 + q);
            sh.above = cum;
            sh.bin = loc[q];
            break;
          }
          cum += loc[q];
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sh.digit) << shift;
    mask |= 255u << shift;
    remaining -= sh.above;
    const int bin = sh.bin;
    __syncthreads();
    if (bin == remaining) {  // the k-th key's bin is taken whole
      sel.thresh = prefix - 1u;
      sel.need = 0;
      return sel;
    }
    if (shift == 0) break;
  }
  sel.thresh = prefix;
  sel.need = remaining;
  return sel;
}

// Writes the selected indices (ascending) to out[0..total) and returns total.  Warp w scans the
// contiguous segment [w*seg, (w+1)*seg) 32 keys at a time (conflict-free shared reads); ranks come
// from ballots, segment offsets from one block scan.
template <int NT>
DSA_DEV int compact_ascending(const uint32_t* keys, int n, const Selection& sel, int32_t* out,
                              SelectScratch<NT>& sh) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = ((n + NW - 1) / NW + 31) & ~31;
  const int lo = min(n, warp * seg), hi = min(n, lo + seg);
  const unsigned below = (1u << lane) - 1u;
  int gt = 0, eq = 0;
  for (int base = lo; base < hi; base += 32) {
    const int j = base + lane;
    const uint32_t key = j < hi ? keys[j] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, key > sel.thresh));
    eq += __popc(__ballot_sync(0xffffffffu, key == sel.thresh && key != 0u));
  }
  // exclusive scans over warps of (eq) and of (selected) counts, in warp order = index order
  if (lane == 0) {
    sh.hist[0][warp] = eq;
    sh.hist[0][NW + warp] = gt;
  }
  __syncthreads();
  int eq_before = 0, sel_before = 0, total = 0;
  for (int w = 0; w < NW; ++w) {
    const int e = sh.hist[0][w];
    const int take = max(0, min(e, sel.need - eq_before));
    const int s = sh.hist[0][NW + w] + take;
    if (w < warp) sel_before += s;
    total += s;
    if (w < warp) eq_before += e;
    else if (w == warp) break;
  }
  // total over all warps (recomputed by every thread, the loop above stops at this warp)
  {
    int eb = 0, t = 0;
    for (int w = 0; w < NW; ++w) {
      const int e = sh.hist[0][w];
      t += sh.hist[0][NW + w] + max(0, min(e, sel.need - eb));
      eb += e;
    }
    total = t;
  }
  int take_eq = max(0, sel.need - eq_before);
  int pos = sel_before;
  for (int base = lo; base < hi; base += 32) {
    const int j = base + lane;
    const uint32_t key = j < hi ? keys[j] : 0u;
    const bool is_gt = key > sel.thresh;
    const bool is_eq = key == sel.thresh && key != 0u;
    const unsigned beq = __ballot_sync(0xffffffffu, is_eq);
    const int eq_rank = __popc(beq & below);
    const bool take = is_gt || (is_eq && eq_rank < take_eq);
    const unsigned bt = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(bt & below)] = j;
    pos += __popc(bt);
    take_eq = max(0, take_eq - __popc(beq));
  }
  __syncthreads();
  return total;
}

// ------------------------------------------------------------------------------ small k
// Top-k for k <= kTopkSmallMaxK with one histogram pass.  The valid keys' scores are binned
// linearly between their min and max (a monotone map: no key in a bin is larger than a key in a
// higher bin; the top tail of a row is sparse, so the bin holding the k-th largest is small), and
// the bin b* holding the k-th largest is found from the bins' suffix sums.  Every
// key in a bin above b* is selected; the keys in b* (the top tail of a row is sparse, so usually a
// handful) are ranked by (key descending, index ascending) and the best `need` of them join.  The
// selection is kept as a bitmap over indices, built with ballots, so the ascending output needs
// only popcounts and one block scan.  Returns -1 (nothing written) when b* holds more than
// kTopkMaxCand keys (heavy ties): the caller then falls back to radix_select +
// compact_ascending, which selects the same set.
constexpr int kTopkSmallMaxK = 256;
constexpr int kTopkMaxCand = 512;
constexpr int kTopkBins = 2048;
constexpr int kTopkMaxN = 32768;

// The score a key came from (score_key inverted; -0 comes back as +0).
DSA_DEV float key_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

struct TopkScratch {
  int hist[kTopkBins];
  int crank[kTopkMaxCand];
  uint32_t bits[kTopkMaxN / 32];
  uint32_t ckey[kTopkMaxCand];
  int cidx[kTopkMaxCand];
  uint32_t wmin[32], wmax[32];
  int wcnt[32];
  int n_cand, strict_above, bstar, red[33];
};

// Count, min and max of the valid keys a thread wrote, reduced inside topk_small.
struct KeyStats {
  int c = 0;
  uint32_t mn = 0xffffffffu, mx = 0u;
  DSA_DEV void add(uint32_t key) {
    if (key != 0u) {
      ++c;
      mn = min(mn, key);
      mx = max(mx, key);
    }
  }
};

// `st`: this thread's share of the key statistics (any partition of the keys over the threads).
// Rank of candidate i among the candidates by (key descending, index ascending): the number of
// candidates ahead of it.  Eight candidates per round, read as shared-memory broadcasts.
DSA_DEV int candidate_rank(const uint32_t* ckey, const int* cidx, int C, uint32_t ki, int ii) {
  int r = 0;
  for (int j0 = 0; j0 < C; j0 += 8) {
    uint32_t kj[8];
    int ij[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = j0 + u < C;
      kj[u] = in ? ckey[j0 + u] : 0u;
      ij[u] = in ? cidx[j0 + u] : 0x7fffffff;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) r += (kj[u] > ki) | ((kj[u] == ki) & (ij[u] < ii));
  }
  return r;
}

// Writes the indices whose bit is set in sh.bits[0, nwords) to out in ascending order (one block
// scan over the words' popcounts); returns their number.
template <int NT>
DSA_DEV int bitmap_to_ascending(int nwords, int32_t* out, TopkScratch& sh) {
  const int tid = threadIdx.x;
  const int per = (nwords + NT - 1) / NT;  // words per thread, contiguous
  const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(sh.bits[w]);
  int total;
  int pos = block_exclusive_scan(cnt, sh.red, &total);
  for (int w = w0; w < w1; ++w) {
    uint32_t word = sh.bits[w];
    while (word) {
      const int b = __ffs(word) - 1;
      out[pos++] = (w << 5) + b;
      word &= word - 1u;
    }
  }
  __syncthreads();
  return total;
}

template <int NT>
DSA_DEV int topk_small(const uint32_t* keys, int n, int k, int32_t* out, TopkScratch& sh,
                       KeyStats st) {
  constexpr int NW = NT / 32;
  static_assert(NT % 32 == 0 && NT >= kTopkBins / 8, "warps, and one thread per 8 bins");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (k <= 0) return 0;
  if (n > kTopkMaxN) return -1;
  const int nwords = (n + 31) >> 5;
  int c = st.c;
  uint32_t mn = st.mn, mx = st.mx;
  c = warp_sum_i(c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sh.wmin[warp] = mn;
    sh.wmax[warp] = mx;
    sh.wcnt[warp] = c;
  }
  for (int b = tid; b < kTopkBins; b += NT) sh.hist[b] = 0;
  if (tid == 0) sh.n_cand = 0;
  __syncthreads();
  int n_valid = 0;
  mn = 0xffffffffu;
  mx = 0u;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    n_valid += sh.wcnt[w];
    mn = min(mn, sh.wmin[w]);
    mx = max(mx, sh.wmax[w]);
  }
  if (n_valid == 0) return 0;
  const float lo = key_score(mn);
  const float span = key_score(mx) - lo;
  const float scale = span > 0.f ? static_cast<float>(kTopkBins) / span : 0.f;
  auto bin_of = [&](uint32_t key) -> int {
    return min(kTopkBins - 1, static_cast<int>((key_score(key) - lo) * scale));
  };
  int bstar = -1, need = 0;  // k >= n_valid: every valid key is selected (bins > -1)
  if (k < n_valid) {
    if (!(scale > 0.f) || !(scale < INFINITY)) return -1;  // all equal, or a span fp32 can't bin
    for (int j0 = tid; j0 < n; j0 += 8 * NT) {
      uint32_t kk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) kk[u] = j0 + u * NT < n ? keys[j0 + u * NT] : 0u;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (kk[u] != 0u) atomicAdd(&sh.hist[bin_of(kk[u])], 1);
    }
    __syncthreads();
    // thread t < 256 owns bins 2047-8t .. 2040-8t (from the top); exclusive prefix over t of the
    // owned counts = keys in the bins above
    int loc[8], sum = 0;
    if (tid < kTopkBins / 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        loc[q] = sh.hist[kTopkBins - 1 - (tid * 8 + q)];
        sum += loc[q];
      }
    }
    int total;
    const int above = block_exclusive_scan(tid < kTopkBins / 8 ? sum : 0, sh.red, &total);
    if (tid < kTopkBins / 8 && above < k && above + sum >= k) {
      int cum = above;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (cum + loc[q] >= k) {
          sh.bstar = kTopkBins - 1 - (tid * 8 + q);
          sh.strict_above = cum;  // keys in bins > b*
          break;
        }
        cum += loc[q];
      }
    }
    __syncthreads();
    bstar = sh.bstar;
    need = k - sh.strict_above;
    if (sh.hist[bstar] > kTopkMaxCand) return -1;
  }
  // bitmap of the keys above b*; the keys of b* gathered as candidates.  Lanes of a warp hold 32
  // consecutive indices, so a ballot is one bitmap word.
  for (int j0 = tid; j0 < (nwords << 5); j0 += 8 * NT) {
    uint32_t kk[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) kk[u] = j0 + u * NT < n ? keys[j0 + u * NT] : 0u;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * NT;
      const int bn = kk[u] != 0u ? bin_of(kk[u]) : -2;
      const unsigned sel = __ballot_sync(0xffffffffu, bn > bstar);
      const unsigned cand = __ballot_sync(0xffffffffu, bn == bstar);
      if (j - lane < (nwords << 5) && lane == 0) sh.bits[j >> 5] = sel;
      if (cand != 0u) {
        int base = 0;
        if (lane == 0) base = atomicAdd(&sh.n_cand, __popc(cand));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (bn == bstar) {
          const int at = base + __popc(cand & ((1u << lane) - 1u));
          sh.ckey[at] = kk[u];
          sh.cidx[at] = j;
        }
      }
    }
  }
  __syncthreads();
  // the best `need` keys of b*, by (key descending, index ascending)
  const int C = sh.n_cand;
  for (int i = tid; i < C; i += NT) {
    const int ii = sh.cidx[i];
    if (candidate_rank(sh.ckey, sh.cidx, C, sh.ckey[i], ii) < need)
      atomicOr(&sh.bits[ii >> 5], 1u << (ii & 31));
  }
  __syncthreads();
  return bitmap_to_ascending<NT>(nwords, out, sh);
}

// Top-k of a small candidate set already in sh.ckey / sh.cidx [0, C) (C <= kTopkMaxCand, keys != 0,
// distinct indices < n <= kTopkMaxN): the k best by (key descending, index ascending), written to
// out in ascending index order.  Returns min(k, C).
template <int NT>
DSA_DEV int topk_candidates(int C, int k, int n, int32_t* out, TopkScratch& sh) {
  const int tid = threadIdx.x;
  if (min(k, C) <= 0) return 0;
  const int nwords = (n + 31) >> 5;
  for (int w = tid; w < nwords; w += NT) sh.bits[w] = 0u;
  __syncthreads();
  for (int i = tid; i < C; i += NT) {
    const uint32_t ki = sh.ckey[i];
    const int ii = sh.cidx[i];
    if (candidate_rank(sh.ckey, sh.cidx, C, ki, ii) < k)
      atomicOr(&sh.bits[ii >> 5], 1u << (ii & 31));
  }
  __syncthreads();
  return bitmap_to_ascending<NT>(nwords, out, sh);
}

// Scratch of select_topk_block: the small-k path and the radix fallback never run at once.
template <int NT>
union SelectAnyScratch {
  TopkScratch small;
  SelectScratch<NT> radix;
};

// Top-k of the keys (valid = != 0) into out[0..k): the selected indices in ascending order, then
// -1 up to k; returns the number selected.  Small k takes the one-pass path when it can.  `st`:
// the statistics of the keys this thread wrote.
template <int NT>
DSA_DEV int select_topk_block(const uint32_t* keys, int n, int k, int32_t* out,
                              SelectAnyScratch<NT>& sh, KeyStats st) {
  int total = k <= kTopkSmallMaxK ? topk_small<NT>(keys, n, k, out, sh.small, st) : -1;
  if (total < 0) {
    __syncthreads();  // the small path's scratch is reused by the radix path
    const Selection sel = radix_select<NT>(keys, n, k, sh.radix);
    total = compact_ascending<NT>(keys, n, sel, out, sh.radix);
  }
  for (int i = max(total, 0) + static_cast<int>(threadIdx.x); i < k; i += NT) out[i] = -1;
  return total;
}

}  // namespace dsa
