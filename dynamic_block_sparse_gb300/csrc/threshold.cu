// PSA progressive threshold selection with fused attention, decided entirely on the device.
//
// One CTA of 8 warps per (request, KV head).  The row's block scores are held in shared memory as
// order-preserving keys.  Blocks are visited a chunk at a time in criticality order (score
// descending, ties to the lower index):
//   1. the next `ch` blocks: each thread takes the largest of its keys; the ch-th largest of those
//      per-thread maxima bounds the ch-th largest key of the row from below (ch distinct keys
//      reach it), so only the few keys at or above it are ranked (one thread per key);
//   2. their page-table entries are read in parallel and the pages fetched with TMA;
//   3. one warp per block computes the block's softmax mass of every query head from Q.K alone;
//   4. one warp walks the chunk in rank order with the stop rule AS_acc / (AS_acc + AS_min) >= tau
//      (log domain; with DSA_PSA_NLEFT the rule weighs AS_min by the blocks left);
//   5. the accepted blocks get the P.V pass, one warp per block.
// No host round trip; a typical row (a handful of blocks) is one chunk.
#include "attn_core.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kThrWarps = 8;
constexpr int kThrThreads = kThrWarps * 32;
constexpr int kMaxChunk = 8;
constexpr uint32_t kThrMergeBytes = kThrWarps * (16 * 128 + 32) * 4;

struct ThrLayout {
  uint32_t keys_off, q_off, mass_off, list_off, cand_off, misc_off, total;
  int chunk;
};

__host__ __device__ inline ThrLayout thr_layout(int page, int n_keys) {
  ThrLayout L;
  const uint32_t stage_bytes = 512u * page;
  int chunk = static_cast<int>(65536u / stage_bytes);
  chunk = chunk < 1 ? 1 : (chunk > kMaxChunk ? kMaxChunk : chunk);
  L.chunk = chunk;
  uint32_t area = stage_bytes * chunk;
  if (area < kThrMergeBytes) area = kThrMergeBytes;  // the warps' states at the end
  area = (area + 1023u) & ~1023u;
  L.keys_off = area;
  L.q_off = L.keys_off + ((static_cast<uint32_t>(n_keys) * 4u + 15u) & ~15u);
  L.mass_off = L.q_off + 16u * kQStride * 2u;
  L.list_off = L.mass_off + kMaxChunk * 16u * 4u;
  L.cand_off = L.list_off + 2u * kMaxChunk * 4u;
  L.misc_off = L.cand_off + kThrWarps * kMaxChunk * 8u;
  L.total = L.misc_off + 64u + 1024u;
  return L;
}

DSA_DEV float log2_add(float a, float b) {
  if (a == -INFINITY) return b;
  if (b == -INFINITY) return a;
  const float mx = fmaxf(a, b);
  return mx + log2f(1.f + exp2f(-fabsf(a - b)));
}

// (key, index) as one 64-bit value ordered by key, then by the LOWER index: the larger value is
// the block visited first.  0 = nothing.
DSA_DEV unsigned long long rank_value(uint32_t key, int j) {
  return key == 0u ? 0ull
                   : (static_cast<unsigned long long>(key) << 32) |
                         (0xffffffffu - static_cast<uint32_t>(j));
}

DSA_DEV unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

__global__ void __launch_bounds__(kThrThreads)
    psa_threshold_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const ThresholdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  __shared__ int s_red[33];
  __shared__ __align__(8) uint64_t bar;
  const KvView& kv = a.kv;
  const int page = kv.p;
  const int row = blockIdx.x;
  const int b = row / kv.Hkv, h = row % kv.Hkv;
  if (kv.streaming != nullptr && kv.streaming[h] != 0) return;
  const int L = request_len(kv, b);
  const int npos = (L + page - 1) / page;
  const int n = min(npos, min(a.score_stride, kv.max_pages));
  const ThrLayout lay = thr_layout(page, kv.max_pages);
  const int chunk = lay.chunk;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + lay.keys_off);
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + lay.q_off);
  float* s_mass = reinterpret_cast<float*>(smem + lay.mass_off);  // [chunk][16] log2 mass
  int32_t* s_ranked = reinterpret_cast<int32_t*>(smem + lay.list_off);  // [chunk] positions
  int32_t* s_phys = s_ranked + kMaxChunk;                                // [chunk] pages
  unsigned long long* s_cand = reinterpret_cast<unsigned long long*>(smem + lay.cand_off);
  int* misc = reinterpret_cast<int*>(smem + lay.misc_off);  // accepted, stop, abort, #cand
  volatile int* abort_flag = misc + 2;
  unsigned long long* s_bound = reinterpret_cast<unsigned long long*>(misc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t stage_bytes = 512u * page;
  const uint32_t smem_base = smem_u32(smem);

  // ---- the row's keys (every load in flight) and the query tile
  const float* srow = a.scores + static_cast<size_t>(row) * a.score_stride;
  int c = 0;
  for (int j0 = tid; j0 < n; j0 += 8 * kThrThreads) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = j0 + u * kThrThreads < n ? srow[j0 + u * kThrThreads] : -INFINITY;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (j0 + u * kThrThreads < n) {
        const uint32_t k = score_key(v[u]);
        keys[j0 + u * kThrThreads] = k;
        c += k != 0u;
      }
  }
  {
    const int r = tid >> 4, cc = tid & 15;  // one 16-byte piece each: 16 rows x 128 dims
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < kv.G)
      v = *reinterpret_cast<const uint4*>(
          a.q + (static_cast<size_t>(b) * kv.Hq + h * kv.G + r) * kHeadDim + cc * 8);
    *reinterpret_cast<uint4*>(sQ + r * kQStride + cc * 8) = v;
  }
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    misc[2] = 0;
  }
  int n_valid;
  block_exclusive_scan(c, s_red, &n_valid);  // contains __syncthreads
  const int total = min(a.cap, n_valid);

  uint32_t qa[8][4];
  load_q_frags(sQ, qa);
  WarpSoftmaxState st;
  state_init(st);
  const float thr = log2f((1.f - a.tau) / a.tau);  // tau == 1 -> -inf: never satisfied
  const bool use_nleft = (a.flags & DSA_PSA_NLEFT) != 0;
  const int tiles = page / 16;
  float lacc = -INFINITY, lmin = INFINITY;  // warp 0, lane g < G: log2 AS_acc, log2 AS_min
  int visited = 0;
  uint32_t phase = 0;
  int32_t* idx_out = a.idx + static_cast<size_t>(row) * a.idx_stride;

  while (visited < total) {
    const int ch = min(chunk, total - visited);
    // ---- 1. the next ch blocks in criticality order
    unsigned long long mine = 0ull;  // this thread's largest remaining (key, index)
    for (int j = tid; j < n; j += kThrThreads) {
      const unsigned long long v = rank_value(keys[j], j);
      mine = v > mine ? v : mine;
    }
    {  // the warp's ch largest thread maxima, then (warp 0) the ch-th largest of all of them
      unsigned long long v = mine;
      for (int r = 0; r < ch; ++r) {
        const unsigned long long w = warp_max_u64(v);
        if (lane == 0) s_cand[warp * kMaxChunk + r] = w;
        if (v == w) v = 0ull;
      }
    }
    if (tid == 0) misc[3] = 0;
    __syncthreads();
    if (warp == 0) {
      unsigned long long v0 = 0ull, v1 = 0ull;
      for (int i = lane; i < kThrWarps * kMaxChunk; i += 32) {
        const unsigned long long v = (i % kMaxChunk) < ch ? s_cand[i] : 0ull;
        if (i < 32) v0 = v;
        else v1 = v;
      }
      unsigned long long w = 0ull;
      for (int r = 0; r < ch; ++r) {
        w = warp_max_u64(v0 > v1 ? v0 : v1);
        if (v0 == w) v0 = 0ull;
        else if (v1 == w) v1 = 0ull;
      }
      if (lane == 0) *s_bound = w;  // the ch-th largest thread maximum (> 0: ch blocks remain)
    }
    __syncthreads();
    const unsigned long long bound = *s_bound;
    // every key at or above the bound is a candidate; a candidate's rank among them places it
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(smem);  // the stage area
    for (int j = tid; j < n; j += kThrThreads) {
      const unsigned long long v = rank_value(keys[j], j);
      if (v != 0ull && v >= bound) {
        const int at = atomicAdd(&misc[3], 1);
        if (at < static_cast<int>(stage_bytes * chunk / 8)) cand[at] = v;
      }
    }
    __syncthreads();
    const int C = min(misc[3], static_cast<int>(stage_bytes * chunk / 8));
    for (int i = tid; i < C; i += kThrThreads) {
      const unsigned long long v = cand[i];
      int rnk = 0;
      for (int q = 0; q < C; ++q) rnk += cand[q] > v;
      if (rnk < ch) s_ranked[rnk] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(v));
    }
    fence_proxy_async_smem();  // the candidates' space is the stage area TMA writes next
    __syncthreads();
    // ---- 2. page-table entries (one thread each), then the TMA loads
    if (tid < ch) {
      const int pos = s_ranked[tid];
      int ph = kv.page_table[static_cast<size_t>(b) * kv.max_pages + pos];
      if (ph < 0 || ph >= kv.num_phys) {
        raise_status(kv.status, DSA_STATUS_BAD_PAGE);
        ph = -1;
      }
      s_phys[tid] = ph;
      keys[pos] = 0u;  // taken
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t bytes = 0;
      for (int cc = 0; cc < ch; ++cc)
        if (s_phys[cc] >= 0) bytes += stage_bytes;
      const uint32_t full = smem_u32(&bar);
      mbar_arrive_expect_tx(full, bytes);
      for (int cc = 0; cc < ch; ++cc) {
        if (s_phys[cc] < 0) continue;
        const uint32_t dst = smem_base + cc * stage_bytes;
        const int row0 = (s_phys[cc] * kv.Hkv + h) * page;
        tma_load_page(dst, &tmK, row0, full);
        tma_load_page(dst + 2 * page * 128, &tmV, row0, full);
      }
    }
    const bool ok_wait = mbar_wait(smem_u32(&bar), phase & 1u, abort_flag, kv.status);
    ++phase;
    if (named_barrier_or(1, kThrThreads, !ok_wait || *abort_flag)) break;

    // ---- 3. per-block softmax mass (log2 units) of every query row, one warp per block
    for (int cc = warp; cc < ch; cc += kThrWarps) {
      float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
      if (s_phys[cc] >= 0) {
        const int pos = s_ranked[cc];
        const uint32_t kb = smem_base + cc * stage_bytes;
        for (int t = 0; t < tiles; ++t) {
          const bool in = pos * page + t * 16 + (lane & 15) < L;
          const uint32_t valid = __ballot_sync(0xffffffffu, in) & 0xffffu;
          if (valid == 0u) continue;
          float sc[2][4];
          tile_scores(qa, kb, page, t * 16, sc);
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
        s_mass[cc * 16 + r0] = mrow[0] == -INFINITY ? -INFINITY : mrow[0] + log2f(lrow[0]);
        s_mass[cc * 16 + r0 + 8] = mrow[1] == -INFINITY ? -INFINITY : mrow[1] + log2f(lrow[1]);
      }
    }
    __syncthreads();

    // ---- 4. stop rule, walked in rank order by warp 0 (lane g tracks query head g)
    if (warp == 0) {
      int accepted = ch, stop = 0;
      for (int cc = 0; cc < ch; ++cc) {
        const float x = s_mass[cc * 16 + (lane & 15)];
        if (lane < kv.G && x > -INFINITY) {
          lacc = log2_add(lacc, x);
          lmin = fminf(lmin, x);
        }
        const int nleft = n_valid - (visited + cc + 1);
        float lhs = lmin - lacc;
        if (use_nleft) lhs += nleft > 0 ? log2f(static_cast<float>(nleft)) : -INFINITY;
        const bool ok = lane >= kv.G || (lacc > -INFINITY && lhs <= thr);
        if (__all_sync(0xffffffffu, ok)) {
          accepted = cc + 1;
          stop = 1;
          break;
        }
      }
      if (lane == 0) {
        misc[0] = accepted;
        misc[1] = stop;
      }
    }
    __syncthreads();
    const int accepted = misc[0];
    const int stop = misc[1];

    // ---- 5. P.V for the accepted blocks, one warp per block
    bool wrote = false;
    for (int cc = warp; cc < accepted; cc += kThrWarps) {
      if (s_phys[cc] < 0) continue;
      const int pos = s_ranked[cc];
      const uint32_t kb = smem_base + cc * stage_bytes;
      const uint32_t vb = kb + 2 * page * 128;
      for (int t = 0; t < tiles; ++t) {
        const bool in = pos * page + t * 16 + (lane & 15) < L;
        const uint32_t valid = __ballot_sync(0xffffffffu, in) & 0xffffu;
        if (valid == 0u) continue;
        if (valid != 0xffffu)
          wrote |= zero_invalid_v_rows(valid, smem + cc * stage_bytes + 2 * page * 128, page,
                                       t * 16);
        float sc[2][4];
        tile_scores(qa, kb, page, t * 16, sc);
        tile_softmax_pv(st, sc, a.scale_log2, valid, vb, page, t * 16);
      }
    }
    if (tid < accepted) idx_out[visited + tid] = s_ranked[tid];
    visited += accepted;
    if (wrote) fence_proxy_async_smem();
    __syncthreads();
    if (stop) break;
  }
  if (tid == 0) a.count[row] = visited;
  state_finish(st);
  __syncthreads();
  if (*abort_flag) {  // a wait gave up: let this chunk's loads land (bounded) before leaving
    if (tid == 0) {
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
  state_store(st, sO + warp * 2048, sM + warp * 16, sL + warp * 16);
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
}

}  // namespace

cudaError_t launch_threshold(const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const ThresholdArgs& a, cudaStream_t s) {
  const ThrLayout lay = thr_layout(a.kv.p, a.kv.max_pages);
  cudaError_t e =
      ensure_dynamic_smem(reinterpret_cast<const void*>(psa_threshold_kernel), lay.total);
  if (e != cudaSuccess) return e;
  psa_threshold_kernel<<<a.kv.B * a.kv.Hkv, kThrThreads, lay.total, s>>>(tmK, tmV, a);
  return cudaGetLastError();
}

size_t threshold_smem_bytes(int page, int max_pages) { return thr_layout(page, max_pages).total; }

}  // namespace dsa
