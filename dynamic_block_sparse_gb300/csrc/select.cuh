// Block-wide top-K selection over order-preserving uint32 keys held in shared memory.
//
// radix_select finds the k-th largest key T with four 8-bit digit passes (histograms built with
// warp-aggregated shared atomics), and how many keys equal to T belong to the top-k (`need`);
// compact_ascending then writes the selected indices in ascending index order, taking the keys
// equal to T at the lowest indices, which is the "ties go to the lower page index" rule.
#pragma once

#include "common.cuh"

namespace dsa {

struct Selection {
  uint32_t thresh;  // keys > thresh are selected
  int need;         // plus this many keys == thresh, lowest indices first
  int n_valid;      // keys != 0
};

// Shared scratch used by the routines below.
struct SelectScratch {
  int hist[256];
  int red[33];
  int digit;
  int above;
};

template <int NT>
DSA_DEV Selection radix_select(const uint32_t* keys, int n, int k, SelectScratch& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int c = 0;
  for (int j = tid; j < n; j += NT) c += keys[j] != 0u;
  int n_valid;
  block_exclusive_scan(c, sh.red, &n_valid);
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
  uint32_t prefix = 0u, mask = 0u;
  int remaining = k;
  const int iters = (n + NT - 1) / NT;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int e = tid; e < 256; e += NT) sh.hist[e] = 0;
    __syncthreads();
    for (int it = 0; it < iters; ++it) {
      const int j = it * NT + tid;
      const uint32_t key = j < n ? keys[j] : 0u;
      const int digit =
          (key != 0u && (key & mask) == prefix) ? static_cast<int>((key >> shift) & 255u) : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, digit);
      if (digit >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255-8l .. 248-8l (from the top); find the bin where the count of keys
      // at or above it first reaches `remaining`.
      int loc[8], s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        loc[q] = sh.hist[255 - (lane * 8 + q)];
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
    __syncthreads();
  }
  sel.thresh = prefix;
  sel.need = remaining;
  return sel;
}

// Writes the selected indices (ascending) to out[0..total) and returns total.
template <int NT>
DSA_DEV int compact_ascending(const uint32_t* keys, int n, const Selection& sel, int32_t* out,
                              SelectScratch& sh) {
  const int tid = threadIdx.x;
  const int seg = (n + NT - 1) / NT;
  const int lo = min(n, tid * seg), hi = min(n, lo + seg);
  int gt = 0, eq = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = keys[j];
    gt += key > sel.thresh;
    eq += (key == sel.thresh && key != 0u);
  }
  int eq_total;
  const int eq_before = block_exclusive_scan(eq, sh.red, &eq_total);
  const int take_eq = max(0, min(eq, sel.need - eq_before));
  int total;
  int pos = block_exclusive_scan(gt + take_eq, sh.red, &total);
  int e = 0;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = keys[j];
    if (key > sel.thresh) {
      out[pos++] = j;
    } else if (key == sel.thresh && key != 0u) {
      if (e < take_eq) out[pos++] = j;
      ++e;
    }
  }
  return total;
}

}  // namespace dsa
