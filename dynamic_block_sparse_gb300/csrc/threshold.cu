// PSA progressive threshold selection with fused attention, decided entirely on the device.
//
// One CTA per (request, KV head).  The row's block scores live in shared memory as order-
// preserving keys.  Blocks are ranked lazily, a chunk at a time: the next `chunk` blocks in
// criticality order are found with a radix select over the keys not yet taken and sorted among
// themselves; their K/V pages are fetched with TMA; every block's softmax mass (per query head)
// is computed from Q.K alone; one warp walks the chunk in rank order applying the stop rule
// AS_acc / (AS_acc + AS_min) >= tau in the log domain; only the accepted blocks then get the
// P.V pass.  No host round trip, and a typical row (a handful of blocks) is one chunk.
#include "attn_core.cuh"
#include "internal.h"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kThrWarps = 4;
constexpr int kThrThreads = kThrWarps * 32;
constexpr int kMaxChunk = 8;
constexpr uint32_t kThrMergeBytes = kThrWarps * (16 * 128 + 32) * 4;

struct ThrLayout {
  uint32_t keys_off, q_off, mass_off, list_off, bar_off, misc_off, total;
  int chunk;
};

__host__ __device__ inline ThrLayout thr_layout(int page, int n_keys) {
  ThrLayout L;
  const uint32_t stage_bytes = 512u * page;
  int chunk = static_cast<int>(65536u / stage_bytes);
  chunk = chunk < 1 ? 1 : (chunk > kMaxChunk ? kMaxChunk : chunk);
  L.chunk = chunk;
  uint32_t area = stage_bytes * chunk;
  if (area < kThrMergeBytes) area = kThrMergeBytes;
  area = (area + 1023u) & ~1023u;
  L.keys_off = area;
  L.q_off = L.keys_off + ((static_cast<uint32_t>(n_keys) * 4u + 15u) & ~15u);
  L.mass_off = L.q_off + 16u * kQStride * 2u;
  L.list_off = L.mass_off + kMaxChunk * 16u * 4u;
  L.bar_off = L.list_off + 3u * kMaxChunk * 4u;
  L.misc_off = L.bar_off + 16u;
  L.total = L.misc_off + 64u + 1024u;
  return L;
}

DSA_DEV float log2_add(float a, float b) {
  if (a == -INFINITY) return b;
  if (b == -INFINITY) return a;
  const float mx = fmaxf(a, b);
  return mx + log2f(1.f + exp2f(-fabsf(a - b)));
}

__global__ void __launch_bounds__(kThrThreads)
    psa_threshold_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const ThresholdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  __shared__ SelectScratch<kThrThreads> sh;
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
  float* s_mass = reinterpret_cast<float*>(smem + lay.mass_off);
  int32_t* s_chunk = reinterpret_cast<int32_t*>(smem + lay.list_off);
  int32_t* s_ranked = s_chunk + kMaxChunk;
  int32_t* s_phys = s_ranked + kMaxChunk;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  int* misc = reinterpret_cast<int*>(smem + lay.misc_off);  // [0] accepted, [1] stop, [2] abort
  volatile int* abort_flag = misc + 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t stage_bytes = 512u * page;
  const uint32_t smem_base = smem_u32(smem);

  const float* srow = a.scores + static_cast<size_t>(row) * a.score_stride;
  int c = 0;
  for (int j = tid; j < n; j += kThrThreads) {
    const uint32_t k = score_key(srow[j]);
    keys[j] = k;
    c += k != 0u;
  }
  for (int e = tid; e < 16 * 16; e += kThrThreads) {
    const int r = e >> 4, cc = e & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < kv.G)
      v = *reinterpret_cast<const uint4*>(
          a.q + (static_cast<size_t>(b) * kv.Hq + h * kv.G + r) * kHeadDim + cc * 8);
    *reinterpret_cast<uint4*>(sQ + r * kQStride + cc * 8) = v;
  }
  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    fence_mbar_init();
    misc[2] = 0;
  }
  int n_valid;
  block_exclusive_scan(c, sh.red, &n_valid);  // contains __syncthreads
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
    const Selection sel = radix_select<kThrThreads>(keys, n, ch, sh);
    compact_ascending<kThrThreads>(keys, n, sel, s_chunk, sh);
    __syncthreads();
    if (warp == 0) {
      const int my_idx = lane < ch ? s_chunk[lane] : -1;
      const uint32_t my_key = lane < ch ? keys[my_idx] : 0u;
      int rank = 0;
      for (int j = 0; j < ch; ++j) {
        const int oj = __shfl_sync(0xffffffffu, my_idx, j);
        const uint32_t ok = __shfl_sync(0xffffffffu, my_key, j);
        rank += (ok > my_key || (ok == my_key && oj < my_idx)) ? 1 : 0;
      }
      if (lane < ch) s_ranked[rank] = my_idx;
    }
    __syncthreads();
    if (tid < ch) keys[s_chunk[tid]] = 0u;
    if (tid == 0) {
      uint32_t bytes = 0;
      for (int cc = 0; cc < ch; ++cc) {
        const int pos = s_ranked[cc];
        int ph = kv.page_table[static_cast<size_t>(b) * kv.max_pages + pos];
        if (ph < 0 || ph >= kv.num_phys) {
          raise_status(kv.status, DSA_STATUS_BAD_PAGE);
          ph = -1;
        } else {
          bytes += stage_bytes;
        }
        s_phys[cc] = ph;
      }
      const uint32_t full = smem_u32(bar);
      mbar_arrive_expect_tx(full, bytes);
      for (int cc = 0; cc < ch; ++cc) {
        if (s_phys[cc] < 0) continue;
        const uint32_t dst = smem_base + cc * stage_bytes;
        const int row0 = (s_phys[cc] * kv.Hkv + h) * page;
        tma_load_page(dst, &tmK, row0, full);
        tma_load_page(dst + 2 * page * 128, &tmV, row0, full);
      }
    }
    __syncthreads();
    const bool ok_wait = mbar_wait(smem_u32(bar), phase & 1u, abort_flag, kv.status);
    ++phase;
    __syncthreads();
    if (!ok_wait || *abort_flag) break;

    // ---- phase A: per-block softmax mass (log2 units) of every query row
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

    // ---- stop rule, walked in rank order by warp 0 (lane g tracks query head g)
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

    // ---- phase B: P.V for the accepted blocks
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
  if (*abort_flag) return;

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
