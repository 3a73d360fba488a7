// PSA progressive threshold selection with fused attention, decided entirely on the device.
//
// One CTA of 8 warps per (request, KV head).  The row's block scores arrive in shared memory with
// one bulk copy and become order-preserving 32-bit keys in place.  Blocks are visited a chunk at
// a time (up to 16) in criticality order (score descending, ties to the lower index):
//   1. the next `ch` blocks: every thread keeps the two largest of its keys; the ch-th largest of
//      the warps' top two keys (16 keys at distinct positions) bounds the ch-th largest key of the
//      row from below, so only the few keys at or above it are ranked;
//   2. one lane per warp completes the chunk's page-table entries (mostly loaded early, as each
//      thread's largest key) and issues the TMA loads of its blocks;
//   3. one warp per block computes the block's softmax mass of every query head from Q.K alone,
//      keeping the Q.K tiles for step 5;
//   4. every warp evaluates the stop rule AS_acc / (AS_acc + AS_min) >= tau after every block of
//      the chunk at once (prefix sums and minima in rank order, the same result in each warp, so
//      that no warp waits for another's; with DSA_PSA_NLEFT the rule weighs AS_min by the blocks
//      left) and accepts up to the first block that meets it;
//   5. the accepted blocks get the P.V pass, one warp per block.
// No host round trip.  A row whose accepted set fits in one chunk costs a single pass; the chunk is
// sized so that typical rows do (blocks past the stop point are fetched and then dropped).
#include "attn_core.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsa {
#ifdef DSA_TIMELINE
__device__ unsigned long long g_trace_threshold[kTraceCtas * 2 * kTraceSlots];
#endif
namespace {

constexpr int kThrWarps = 8;
constexpr int kThrThreads = kThrWarps * 32;
constexpr int kMaxChunk = 16;                     // blocks per chunk (and lanes per head slot)
constexpr uint32_t kThrStageBudget = 131072u;     // bytes of staged pages per chunk
constexpr uint32_t kThrSmemLimit = 227u * 1024u;  // dynamic shared memory a CTA may hold
constexpr uint32_t kThrMergeBytes = kThrWarps * (16 * 128 + 32) * 4;

struct ThrLayout {
  uint32_t keys_off, q_off, mass_off, pacc_off, pmin_off, state_off, list_off, misc_off, sc_off,
      total;
  int chunk;
};

__host__ __device__ inline ThrLayout thr_layout_for(int page, int n_keys, int chunk) {
  ThrLayout L;
  const uint32_t stage_bytes = 512u * page;
  L.chunk = chunk;
  uint32_t area = stage_bytes * chunk;
  if (area < kThrMergeBytes) area = kThrMergeBytes;  // the warps' states at the end
  area = (area + 1023u) & ~1023u;
  L.keys_off = area;
  // the score row lands with its global 16-byte phase (up to 12 bytes in), then becomes keys
  L.q_off = L.keys_off + ((static_cast<uint32_t>(n_keys) * 4u + 16u + 15u) & ~15u);
  L.mass_off = L.q_off + 16u * kQStride * 2u;
  L.pacc_off = L.mass_off + kMaxChunk * 16u * 4u;
  L.pmin_off = L.pacc_off + kMaxChunk * 16u * 4u;
  L.state_off = L.pmin_off + kMaxChunk * 16u * 4u;
  L.list_off = L.state_off + 64u * 4u;
  L.misc_off = L.list_off + 2u * kMaxChunk * 4u;
  L.sc_off = L.misc_off + 64u;
  // the chunk's Q.K tiles as mma fragments (1 KB per 16-token tile), reused by the P.V pass
  L.total = L.sc_off + static_cast<uint32_t>(chunk) * (page / 16) * 1024u + 1024u;
  return L;
}

// The largest chunk (up to kMaxChunk blocks and kThrStageBudget bytes of pages) whose layout fits.
__host__ __device__ inline ThrLayout thr_layout(int page, int n_keys) {
  int chunk = static_cast<int>(kThrStageBudget / (512u * page));
  chunk = chunk < 1 ? 1 : (chunk > kMaxChunk ? kMaxChunk : chunk);
  ThrLayout L = thr_layout_for(page, n_keys, chunk);
  while (L.total > kThrSmemLimit && chunk > 1) {
    chunk >>= 1;
    L = thr_layout_for(page, n_keys, chunk);
  }
  return L;
}

// (key, index) as one 64-bit value ordered by key, then by the LOWER index: the larger value is
// the block visited first.  0 = nothing.
DSA_DEV unsigned long long rank_value(uint32_t key, int j) {
  return key == 0u ? 0ull
                   : (static_cast<unsigned long long>(key) << 32) |
                         (0xffffffffu - static_cast<uint32_t>(j));
}

DSA_DEV int rank_pos(unsigned long long v) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(v));
}

// Page id not looked up yet (a table entry with this value is invalid anyway).
constexpr int32_t kPhysUnknown = INT32_MIN;

constexpr int kScanUnroll = 16;  // keys a thread loads at once

// The two largest keys over this thread's positions j = tid, tid + 256, ... (< n) (a key held at
// two positions counts twice) and the lowest position holding the largest: sixteen loads in
// flight per pass, then a pairwise max/min tree.  kConvert: the entries are still the float
// scores (keys[] is their in-place view): convert them, store the keys and count the valid ones.
template <bool kConvert>
DSA_DEV void thread_top2(uint32_t* keys, int n, int tid, uint32_t& first, uint32_t& second,
                         int& jfirst, int& count) {
  first = second = 0u;
  jfirst = 0;
  for (int j0 = 0; j0 < n; j0 += kScanUnroll * kThrThreads) {
    uint32_t k[kScanUnroll];
#pragma unroll
    for (int u = 0; u < kScanUnroll; ++u) {
      // the load's index is clamped rather than guarded, so that all sixteen issue at once
      const int j = j0 + u * kThrThreads + tid;
      const uint32_t raw = keys[min(j, n - 1)];
      k[u] = j < n ? (kConvert ? score_key(__uint_as_float(raw)) : raw) : 0u;
      if (kConvert) {
        if (j < n) keys[j] = k[u];
        count += k[u] != 0u;
      }
    }
    uint32_t f[kScanUnroll / 2], s[kScanUnroll / 2];
#pragma unroll
    for (int u = 0; u < kScanUnroll / 2; ++u) {
      f[u] = max(k[2 * u], k[2 * u + 1]);
      s[u] = min(k[2 * u], k[2 * u + 1]);
    }
#pragma unroll
    for (int w = kScanUnroll / 4; w >= 1; w >>= 1)
#pragma unroll
      for (int u = 0; u < w; ++u) {
        const uint32_t f1 = f[2 * u], f2 = f[2 * u + 1];
        const uint32_t s1 = s[2 * u], s2 = s[2 * u + 1];
        f[u] = max(f1, f2);
        s[u] = max(min(f1, f2), max(s1, s2));
      }
    int jp = 0;
#pragma unroll
    for (int u = kScanUnroll - 1; u >= 0; --u)
      if (k[u] == f[0]) jp = j0 + u * kThrThreads + tid;
    if (f[0] > first) jfirst = jp;  // equal keys keep the earlier (lower) position
    second = max(min(first, f[0]), max(second, s[0]));
    first = max(first, f[0]);
  }
}

// Largest 64-bit value held by the warp's lanes: the high words first, then the low words among
// the lanes holding the largest high word (two 32-bit warp reductions).
DSA_DEV unsigned long long warp_max_u64(unsigned long long v) {
  const uint32_t hi = static_cast<uint32_t>(v >> 32), lo = static_cast<uint32_t>(v);
  const uint32_t whi = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t wlo = __reduce_max_sync(0xffffffffu, hi == whi ? lo : 0u);
  return (static_cast<unsigned long long>(whi) << 32) | wlo;
}

__global__ void __launch_bounds__(kThrThreads)
    psa_threshold_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const ThresholdArgs a) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  __shared__ int s_red[kThrWarps];              // valid keys per warp
  __shared__ uint32_t s_wtop[2 * kThrWarps];     // each warp's two largest keys
  __shared__ __align__(8) uint64_t bar, bar_keys;
  const KvView& kv = a.kv;
  const int page = kv.p;
  const int row = blockIdx.x;
  const int b = row / kv.Hkv, h = row % kv.Hkv;
  const ThrLayout lay = thr_layout(page, kv.max_pages);
  const int chunk = lay.chunk;
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + lay.q_off);
  float* s_mass = reinterpret_cast<float*>(smem + lay.mass_off);  // [chunk][16] log2 mass
  float* s_pacc = reinterpret_cast<float*>(smem + lay.pacc_off);  // [chunk][16] prefix AS_acc
  float* s_pmin = reinterpret_cast<float*>(smem + lay.pmin_off);  // [chunk][16] prefix minima
  // log2 AS_acc and AS_min [2][16] each, alternating by chunk: every warp evaluates the stop rule,
  // so the state a chunk reads is never the one it writes
  float* s_lacc = reinterpret_cast<float*>(smem + lay.state_off);
  float* s_lmin = s_lacc + 32;
  float* s_sc = reinterpret_cast<float*>(smem + lay.sc_off);
  int32_t* s_ranked = reinterpret_cast<int32_t*>(smem + lay.list_off);  // [chunk] positions
  int32_t* s_phys = s_ranked + kMaxChunk;                                // [chunk] pages
  int* misc = reinterpret_cast<int*>(smem + lay.misc_off);  // [2] abort flag, [3] #candidates
  volatile int* abort_flag = misc + 2;
  unsigned long long* s_bound = reinterpret_cast<unsigned long long*>(misc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t stage_bytes = 512u * page;
  const uint32_t smem_base = smem_u32(smem);
  DSA_TRACE_BEGIN();

  // ---- the row's scores: one bulk copy of the whole row, issued before anything else and not
  // waiting for the request length (the unaligned head and tail, at most 3 floats each, by plain
  // loads); the query tile, the request length and the streaming flag load meanwhile
  const float* srow = a.scores + static_cast<size_t>(row) * a.score_stride;
  const int nload = min(a.score_stride, kv.max_pages);
  const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(srow)) & 15u;
  float* fkeys = reinterpret_cast<float*>(smem + lay.keys_off + mis);  // srow's 16-byte phase
  uint32_t* keys = reinterpret_cast<uint32_t*>(fkeys);  // converted in place
  const int head = min(nload, static_cast<int>(((16u - mis) & 15u) >> 2));
  const int body = (nload - head) & ~3;
  const int tail0 = head + body;
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    mbar_init(smem_u32(&bar), kThrWarps);  // every warp arrives once per chunk
    mbar_init(smem_u32(&bar_keys), 1);
    fence_mbar_init();
    misc[2] = 0;
    if (body > 0) {
      mbar_arrive_expect_tx(smem_u32(&bar_keys), static_cast<uint32_t>(body) * 4u);
      bulk_load(smem_u32(fkeys + head), srow + head, static_cast<uint32_t>(body) * 4u,
                smem_u32(&bar_keys));
    } else {
      mbar_arrive(smem_u32(&bar_keys));
    }
  }
  if (tid >= 32 && tid < 32 + head) fkeys[tid - 32] = srow[tid - 32];
  if (tid >= 64 && tid < 64 + nload - tail0) fkeys[tail0 + tid - 64] = srow[tail0 + tid - 64];
  const bool streaming = kv.streaming != nullptr && kv.streaming[h] != 0;
  const int L = request_len(kv, b);
  {
    const int r = tid >> 4, cc = tid & 15;  // one 16-byte piece each: 16 rows x 128 dims
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < kv.G)
      v = *reinterpret_cast<const uint4*>(
          a.q + (static_cast<size_t>(b) * kv.Hq + h * kv.G + r) * kHeadDim + cc * 8);
    *reinterpret_cast<uint4*>(sQ + r * kQStride + cc * 8) = v;
  }
  if (tid < 32) {
    s_lacc[tid] = -INFINITY;
    s_lmin[tid] = INFINITY;
  }
  __syncthreads();  // barriers initialised, head and tail stored
  const bool keys_ok = mbar_wait(smem_u32(&bar_keys), 0u, abort_flag, kv.status);
  if (named_barrier_or(1, kThrThreads, !keys_ok)) {
    if (tid == 0) {  // let the row's copy land (bounded) before leaving
      const unsigned long long t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(&bar_keys), 0u))
        if (global_timer_ns() - t0 > 50000000ull) break;
    }
    return;
  }
  DSA_STAMP(1);           // the score row has landed
  if (streaming) return;  // the streaming path serves this head
  const int npos = (L + page - 1) / page;
  const int n = min(npos, nload);
  // keys in place; each thread's two largest keys serve the first chunk
  int c = 0, jmine;
  uint32_t mine, second;
  thread_top2<true>(keys, n, tid, mine, second, jmine, c);
  // the page-table entry of this thread's largest key, loaded now and used once the chunk is
  // ranked (most of a chunk's blocks are some thread's largest key)
  DSA_STAMP(2);  // keys converted
  const int32_t* pt_row = kv.page_table + static_cast<size_t>(b) * kv.max_pages;
  int my_phys = mine != 0u ? pt_row[jmine] : kPhysUnknown;
  {
    const int wc = __reduce_add_sync(0xffffffffu, c);  // summed after the first chunk's barrier
    if (lane == 0) s_red[warp] = wc;
  }

  uint32_t qa[8][4];
  load_q_frags(sQ, qa);
  WarpSoftmaxState st;
  state_init(st);
  const float thr = log2f((1.f - a.tau) / a.tau);  // tau == 1 -> -inf: never satisfied
  const bool use_nleft = (a.flags & DSA_PSA_NLEFT) != 0;
  const int tiles = page / 16;
  int visited = 0, n_valid = -1, total = 0;
  uint32_t phase = 0;
  int32_t* idx_out = a.idx + static_cast<size_t>(row) * a.idx_stride;

  while (true) {
    // ---- 1. the next ch blocks in criticality order.  A lower bound on the ch-th largest remaining
    // key: the ch-th largest of the warps' top two keys (16 keys at distinct positions, so at
    // least ch keys reach it), or, when fewer than ch of those are valid or the row is long, the
    // exact ch-th largest of the 256 thread maxima.  Every key at or above the bound is a
    // candidate; a candidate's rank among the candidates places it.
    if (visited > 0) {
      thread_top2<false>(keys, n, tid, mine, second, jmine, c);
      my_phys = mine != 0u ? pt_row[jmine] : kPhysUnknown;
    }
    // the stage area holds the 256 thread maxima (when needed), then the candidates and their
    // page ids
    unsigned long long* s_tmax = reinterpret_cast<unsigned long long*>(smem);
    const int cand_cap = static_cast<int>((stage_bytes * chunk - kThrThreads * 8u) / 12u);
    unsigned long long* cand = s_tmax + kThrThreads;
    int32_t* cand_phys = reinterpret_cast<int32_t*>(cand + cand_cap);
    {
      const uint32_t w1 = __reduce_max_sync(0xffffffffu, mine);
      const int at_top = __popc(__ballot_sync(0xffffffffu, mine == w1));
      const uint32_t w2 =
          at_top >= 2 ? w1 : __reduce_max_sync(0xffffffffu, mine == w1 ? second : mine);
      if (lane == 0) {
        s_wtop[2 * warp] = w1;
        s_wtop[2 * warp + 1] = w2;
      }
    }
    if (tid == 0) misc[3] = 0;
    __syncthreads();
    if (n_valid < 0) {  // first pass: the row's valid blocks
      n_valid = 0;
#pragma unroll
      for (int w = 0; w < kThrWarps; ++w) n_valid += s_red[w];
      total = min(a.cap, n_valid);
    }
    DSA_STAMP(3);  // warp keys shared
    if (visited >= total) break;
    const int ch = min(chunk, total - visited);
    unsigned long long bound = 0ull;  // candidates: rank values at or above it
    bool exact = n > cand_cap;
    if (!exact) {  // every warp ranks the 16 warp keys itself (no further barrier)
      const uint32_t mv = lane < 2 * kThrWarps ? s_wtop[lane] : 0u;
      int gt = 0, ge = 0;
#pragma unroll
      for (int k = 0; k < 2 * kThrWarps; ++k) {
        const uint32_t o = __shfl_sync(0xffffffffu, mv, k);
        gt += o > mv;
        ge += o >= mv;
      }
      const uint32_t sel =
          __ballot_sync(0xffffffffu, lane < 2 * kThrWarps && mv != 0u && gt < ch && ge >= ch);
      if (sel != 0u) bound = static_cast<unsigned long long>(__shfl_sync(0xffffffffu, mv, __ffs(sel) - 1)) << 32;
      else exact = true;
    }
    if (exact) {  // uniform: the exact ch-th largest thread maximum (warp 0)
      s_tmax[tid] = rank_value(mine, jmine);
      __syncthreads();
      if (warp == 0) {
        unsigned long long v[kThrThreads / 32], lm = 0ull;
#pragma unroll
        for (int i = 0; i < kThrThreads / 32; ++i) {
          v[i] = s_tmax[i * 32 + lane];
          lm = v[i] > lm ? v[i] : lm;
        }
        unsigned long long w = 0ull;
#pragma unroll 1
        for (int r = 0; r < ch; ++r) {
          w = warp_max_u64(lm);
          if (lm == w) {  // values are distinct (the index is in the low word) unless 0
            lm = 0ull;
#pragma unroll
            for (int i = 0; i < kThrThreads / 32; ++i) {
              if (v[i] == w) v[i] = 0ull;
              lm = v[i] > lm ? v[i] : lm;
            }
          }
        }
        // 0 when fewer than ch threads hold keys: then every remaining key is a candidate, at
        // most (ch - 1) x n / 256 of them
        if (lane == 0) *s_bound = w;
      }
      __syncthreads();
      bound = *s_bound;
    }
    DSA_STAMP(4);  // bound
    // every thread checks its own keys against the bound (sixteen loads in flight, compared as
    // 32-bit words) and each warp claims the slots of its hits with one atomic; only the key
    // positions where some lane of the warp hit are then visited.  A hit that is the thread's
    // largest key brings the page id loaded early.
    const unsigned long long vmine = rank_value(mine, jmine);
    const uint32_t bhi = static_cast<uint32_t>(bound >> 32), blo = static_cast<uint32_t>(bound);
    for (int j0 = 0; j0 < n; j0 += kScanUnroll * kThrThreads) {
      uint32_t hit = 0u;
#pragma unroll
      for (int u = 0; u < kScanUnroll; ++u) {
        const int j = j0 + u * kThrThreads + tid;
        const uint32_t kk = keys[min(j, n - 1)];
        const bool h = (j < n) & (kk != 0u) &
                       ((kk > bhi) | ((kk == bhi) & (0xffffffffu - static_cast<uint32_t>(j) >= blo)));
        hit |= static_cast<uint32_t>(h) << u;
      }
      const uint32_t whit = __reduce_or_sync(0xffffffffu, hit);
      if (whit == 0u) continue;
      const int wtot = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(__popc(hit)));
      int base = 0;
      if (lane == 0) base = atomicAdd(&misc[3], wtot);
      int at = __shfl_sync(0xffffffffu, base, 0);
      for (uint32_t rest = whit; rest != 0u; rest &= rest - 1u) {
        const int u = __ffs(rest) - 1;
        const bool hu = (hit >> u) & 1u;
        const uint32_t bal = __ballot_sync(0xffffffffu, hu);
        const int pos = at + __popc(bal & ((1u << lane) - 1u));
        if (hu && pos < cand_cap) {
          const int j = j0 + u * kThrThreads + tid;
          const unsigned long long v = rank_value(keys[j], j);
          cand[pos] = v;
          cand_phys[pos] = v == vmine ? my_phys : kPhysUnknown;
        }
        at += __popc(bal);
      }
    }
    __syncthreads();
    DSA_STAMP(5);  // candidates collected
    const int C = min(misc[3], cand_cap);
    // ranks: eight threads per candidate, each counting a strided eighth of the candidates above it
    for (int i0 = 0; i0 < C; i0 += kThrThreads / 8) {
      const int i = i0 + (tid >> 3), part = tid & 7;
      int cnt = 0;
      unsigned long long v = 0ull;
      if (i < C) {
        v = cand[i];
#pragma unroll 4
        for (int q = part; q < C; q += 8) cnt += cand[q] > v;
      }
      cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, 4);
      if (part == 0 && i < C && cnt < ch) {
        s_ranked[cnt] = rank_pos(v);
        s_phys[cnt] = cand_phys[i];
      }
    }
    fence_proxy_async_smem();  // the candidates' space is the stage area TMA writes next
    __syncthreads();
    DSA_STAMP(6);  // ranked
    // ---- 2. blocks w and w + 8 of the chunk are warp w's: lane 0 completes their page-table entries
    // and issues their TMA loads (the warps issue in parallel), posting the bytes before its one
    // arrival per chunk
    if (lane == 0) {
      const uint32_t full = smem_u32(&bar);
      for (int cc = warp; cc < ch; cc += kThrWarps) {
        const int pos = s_ranked[cc];
        int ph = s_phys[cc];
        if (ph == kPhysUnknown) ph = pt_row[pos];  // (a table entry equal to it is invalid too)
        if (ph < 0 || ph >= kv.num_phys) {
          raise_status(kv.status, DSA_STATUS_BAD_PAGE);
          ph = -1;
        }
        s_phys[cc] = ph;
        keys[pos] = 0u;  // taken
        if (ph >= 0) {
          mbar_expect_tx(full, stage_bytes);
          const uint32_t dst = smem_base + cc * stage_bytes;
          const int row0 = (ph * kv.Hkv + h) * page;
          tma_load_page(dst, &tmK, row0, full);
          tma_load_page(dst + 2 * page * 128, &tmV, row0, full);
        }
      }
      mbar_arrive(full);
    }
    DSA_STAMP(7);  // TMA issued
    const bool ok_wait = mbar_wait(smem_u32(&bar), phase & 1u, abort_flag, kv.status);
    ++phase;
    if (named_barrier_or(1, kThrThreads, !ok_wait || *abort_flag)) break;
    DSA_STAMP(8);  // pages landed

    // ---- 3. per-block softmax mass (log2 units) of every query row, one warp per block
    for (int cc = warp; cc < ch; cc += kThrWarps) {
      float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
      if (s_phys[cc] >= 0) {
        const int pos = s_ranked[cc];
        const uint32_t kb = smem_base + cc * stage_bytes;
#pragma unroll 1
        for (int t = 0; t < tiles; ++t) {
          const bool in = pos * page + t * 16 + (lane & 15) < L;
          const uint32_t valid = __ballot_sync(0xffffffffu, in) & 0xffffu;
          if (valid == 0u) continue;
          float sc[2][4];
          tile_scores(qa, kb, page, t * 16, sc);
          float4* keep = reinterpret_cast<float4*>(s_sc + ((cc * tiles + t) * 32 + lane) * 8);
          keep[0] = make_float4(sc[0][0], sc[0][1], sc[0][2], sc[0][3]);
          keep[1] = make_float4(sc[1][0], sc[1][1], sc[1][2], sc[1][3]);
          float x[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
              x[nt][e] = ((valid >> col) & 1u) ? sc[nt][e] * a.scale_log2 : -INFINITY;
            }
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float mx = fmaxf(fmaxf(x[0][2 * r], x[0][2 * r + 1]), fmaxf(x[1][2 * r], x[1][2 * r + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(mrow[r], mx);
            float add = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) add += fast_exp2(x[nt][2 * r + e] - mn);
            lrow[r] = lrow[r] * fast_exp2(mrow[r] - mn) + add;
            mrow[r] = mn;
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
          lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
        }
      }
      if ((lane & 3) == 0) {
        const int r0 = lane >> 2;
        s_mass[cc * 16 + r0] = mrow[0] == -INFINITY ? -INFINITY : mrow[0] + fast_log2(lrow[0]);
        s_mass[cc * 16 + r0 + 8] = mrow[1] == -INFINITY ? -INFINITY : mrow[1] + fast_log2(lrow[1]);
      }
    }
    __syncthreads();

    DSA_STAMP(9);  // masses
    // ---- 4. stop rule.  AS_acc and AS_min after each block of the chunk (in rank order) are prefix
    // sums / minima over the chunk on top of the state before it, scanned with lane
    // (head slot gl, block cc) = (lane / 16, lane % 16), two query heads per round; the chunk's
    // accepted prefix ends at the first block after which every head meets the rule.  The sums
    // run in the linear domain relative to the largest term of the head's chunk (one exp2 and one
    // log2 per lane).  Every warp evaluates the rule itself on the same inputs in the same order
    // (so all reach the same decision) rather than one warp deciding while the others wait.
    int accepted, stop;
    {
      const float* lacc_in = s_lacc + ((phase - 1u) & 1u) * 16;
      const float* lmin_in = s_lmin + ((phase - 1u) & 1u) * 16;
      const int cc = lane & (kMaxChunk - 1), gl = lane / kMaxChunk;
      uint32_t okmask = 0xffffu;  // bit cc: every head so far meets the rule after block cc
#pragma unroll 1
      for (int g0 = 0; g0 < kv.G; g0 += 32 / kMaxChunk) {
        const int g = g0 + gl;
        const bool act = g < kv.G && cc < ch;
        const float x = act ? s_mass[cc * 16 + g] : -INFINITY;
        const float acc0 = g < kv.G ? lacc_in[g] : -INFINITY;
        const float min0 = g < kv.G ? lmin_in[g] : INFINITY;
        float ref = fmaxf(x, acc0);
#pragma unroll
        for (int o = 1; o < kMaxChunk; o <<= 1)
          ref = fmaxf(ref, __shfl_xor_sync(0xffffffffu, ref, o));
        float e = x > -INFINITY ? fast_exp2(x - ref) : 0.f;
        float mn = x > -INFINITY ? x : INFINITY;
#pragma unroll
        for (int o = 1; o < kMaxChunk; o <<= 1) {
          const float ye = __shfl_up_sync(0xffffffffu, e, o, kMaxChunk);
          const float ym = __shfl_up_sync(0xffffffffu, mn, o, kMaxChunk);
          if (cc >= o) {
            e += ye;
            mn = fminf(mn, ym);
          }
        }
        const float tot = e + (acc0 > -INFINITY ? fast_exp2(acc0 - ref) : 0.f);
        const float acc = tot > 0.f ? ref + fast_log2(tot) : -INFINITY;
        mn = fminf(min0, mn);
        const int nleft = n_valid - (visited + cc + 1);
        float lhs = mn - acc;
        if (use_nleft) lhs += nleft > 0 ? fast_log2(static_cast<float>(nleft)) : -INFINITY;
        const bool ok = !act || (acc > -INFINITY && lhs <= thr);
        const uint32_t bal = __ballot_sync(0xffffffffu, ok);
        okmask &= bal & (bal >> 16);
        if (act) {  // the running state after block cc (the same values from every warp)
          s_pacc[cc * 16 + g] = acc;
          s_pmin[cc * 16 + g] = mn;
        }
      }
      okmask &= (1u << ch) - 1u;  // ch <= 16
      accepted = okmask != 0u ? __ffs(okmask) : ch;
      stop = okmask != 0u;
      __syncwarp();
      if (lane < kv.G) {
        s_lacc[(phase & 1u) * 16 + lane] = s_pacc[(accepted - 1) * 16 + lane];
        s_lmin[(phase & 1u) * 16 + lane] = s_pmin[(accepted - 1) * 16 + lane];
      }
    }

    DSA_STAMP(10);  // stop decided
    // ---- 5. P.V for the accepted blocks, one warp per block
    bool wrote = false;
    for (int cc = warp; cc < accepted; cc += kThrWarps) {
      if (s_phys[cc] < 0) continue;
      const int pos = s_ranked[cc];
      const uint32_t kb = smem_base + cc * stage_bytes;
      const uint32_t vb = kb + 2 * page * 128;
#pragma unroll 1
      for (int t = 0; t < tiles; ++t) {
        const bool in = pos * page + t * 16 + (lane & 15) < L;
        const uint32_t valid = __ballot_sync(0xffffffffu, in) & 0xffffu;
        if (valid == 0u) continue;
        if (valid != 0xffffu)
          wrote |= zero_invalid_v_rows(valid, smem + cc * stage_bytes + 2 * page * 128, page,
                                       t * 16);
        const float4* keep =
            reinterpret_cast<const float4*>(s_sc + ((cc * tiles + t) * 32 + lane) * 8);
        const float4 k0 = keep[0], k1 = keep[1];
        float sc[2][4] = {{k0.x, k0.y, k0.z, k0.w}, {k1.x, k1.y, k1.z, k1.w}};
        tile_softmax_pv(st, sc, a.scale_log2, valid, vb, page, t * 16);
      }
    }
    if (tid < accepted) idx_out[visited + tid] = s_ranked[tid];
    visited += accepted;
    DSA_STAMP(11);  // P.V (thread 0's warp)
    if (wrote) fence_proxy_async_smem();
    __syncthreads();
    DSA_STAMP(12);  // chunk done
    if (stop || visited >= total) break;
  }
  if (tid == 0) a.count[row] = visited;
  state_finish(st);
  __syncthreads();
  if (*abort_flag) {  // a wait gave up: let this chunk's loads land (bounded) before leaving
    if (tid == 0 && phase > 0u) {
      const unsigned long long t0 = global_timer_ns();
      while (!mbar_try_wait(smem_u32(&bar), (phase - 1u) & 1u))
        if (global_timer_ns() - t0 > 50000000ull) break;
    }
    return;
  }

  // ---- the warps' states merged into the output rows
  float* sO = reinterpret_cast<float*>(smem);
  float* sM = sO + kThrWarps * 2048;
  float* sL = sM + kThrWarps * 16;
  state_store(st, sO + warp * 2048, sM + warp * 16, sL + warp * 16, kv.G);
  __syncthreads();
  for (int e = tid; e < kv.G * kHeadDim; e += kThrThreads) {
    const int g = e >> 7, d = e & 127;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kThrWarps; ++w) M = fmaxf(M, sM[w * 16 + g]);
    float Lsum = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kThrWarps; ++w) {
        const float mw = sM[w * 16 + g];
        if (mw == -INFINITY) continue;
        const float f = fast_exp2(mw - M);
        Lsum += sL[w * 16 + g] * f;
        acc += sO[w * 2048 + g * 128 + d] * f;
      }
    }
    const size_t qh = static_cast<size_t>(b) * kv.Hq + h * kv.G + g;
    a.out[qh * kHeadDim + d] = Lsum > 0.f ? acc / Lsum : 0.f;
    if (d == 0) {
      a.m[qh] = M == -INFINITY ? -INFINITY : M * kLn2;
      a.l[qh] = Lsum;
    }
  }
  DSA_STAMP(13);  // merged and written
  DSA_TRACE_END(g_trace_threshold);
}

}  // namespace

cudaError_t launch_threshold(const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const ThresholdArgs& a, cudaStream_t s) {
  const ThrLayout lay = thr_layout(a.kv.p, a.kv.max_pages);
  cudaError_t e =
      ensure_dynamic_smem(reinterpret_cast<const void*>(psa_threshold_kernel), lay.total);
  if (e != cudaSuccess) return e;
  return launch_pdl(psa_threshold_kernel, a.kv.B * a.kv.Hkv, kThrThreads, lay.total, s, tmK, tmV,
                    a);
}

size_t threshold_smem_bytes(int page, int max_pages) { return thr_layout(page, max_pages).total; }

}  // namespace dsa

#ifdef DSA_TIMELINE
// Phase-trace accessors of the traced library (see DSA_TRACE_BEGIN).
extern "C" int dsa_trace_read_threshold(void* host, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(
      host, dsa::g_trace_threshold, bytes < sizeof(dsa::g_trace_threshold) ? bytes : sizeof(dsa::g_trace_threshold)));
}
extern "C" int dsa_trace_clear_threshold() {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, dsa::g_trace_threshold);
  return static_cast<int>(e == cudaSuccess ? cudaMemset(p, 0, sizeof(dsa::g_trace_threshold)) : e);
}
#endif
