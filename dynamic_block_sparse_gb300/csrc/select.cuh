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

}  // namespace dsa
