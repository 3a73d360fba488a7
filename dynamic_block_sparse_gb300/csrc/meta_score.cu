// Per-page key metadata and page criticality scoring.  Both are streaming HBM scans: 16-byte
// vector loads, several independent loads in flight per thread, no shared-memory staging needed.
#include "common.cuh"
#include "internal.h"
#include "score_core.cuh"

namespace dsa {
namespace {

// ------------------------------------------------------------------------------------ metadata
// 16 bytes of a K row: through the read-only path, or through L2 when the row was written by the
// same kernel (the read-only path is not coherent with such writes).
template <bool COHERENT>
DSA_DEV uint4 ld16(const __nv_bfloat16* p) {
  return COHERENT ? __ldcg(reinterpret_cast<const uint4*>(p))
                  : __ldg(reinterpret_cast<const uint4*>(p));
}

// Metadata of every logical sub-page of page position j of request b (length L), KV head h, on
// physical page phys, computed by one warp.  Lane l reads 16-byte chunk (l & 15) of token rows of
// parity (l >> 4); the two half-warps are combined at the end of every logical page.  The build
// and the append share it, so both write the same bits.
template <int KIND, bool COHERENT>
DSA_DEV void page_meta(const KvView& kv, const __nv_bfloat16* __restrict__ k_pages, int lp,
                       void* __restrict__ meta, int j, int h, int phys, int L, int lane) {
  const int page = kv.p;
  const int valid = min(page, L - j * page);
  const int g = page / lp;
  const int half = lane >> 4, c = lane & 15;
  const __nv_bfloat16* base =
      k_pages + (static_cast<size_t>(phys) * kv.Hkv + h) * page * kHeadDim + c * 8;

  for (int sub = 0; sub < g; ++sub) {
    const int t_lo = sub * lp, t_hi = min((sub + 1) * lp, valid);
    float a[8], bmin[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      a[e] = (KIND == DSA_META_MINMAX) ? -INFINITY : 0.f;
      bmin[e] = INFINITY;
    }
    int t = t_lo + half;
#pragma unroll 1
    for (; t + 6 < t_hi; t += 8) {
      uint4 raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        raw[u] = ld16<COHERENT>(base + static_cast<size_t>(t + 2 * u) * kHeadDim);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&raw[u]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = __bfloat162float(v[e]);
          if (KIND == DSA_META_MINMAX) {
            a[e] = fmaxf(a[e], x);
            bmin[e] = fminf(bmin[e], x);
          } else {
            a[e] += x;
          }
        }
      }
    }
    for (; t < t_hi; t += 2) {
      const uint4 raw = ld16<COHERENT>(base + static_cast<size_t>(t) * kHeadDim);
      const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = __bfloat162float(v[e]);
        if (KIND == DSA_META_MINMAX) {
          a[e] = fmaxf(a[e], x);
          bmin[e] = fminf(bmin[e], x);
        } else {
          a[e] += x;
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float oa = __shfl_xor_sync(0xffffffffu, a[e], 16);
      const float ob = __shfl_xor_sync(0xffffffffu, bmin[e], 16);
      if (KIND == DSA_META_MINMAX) {
        a[e] = fmaxf(a[e], oa);
        bmin[e] = fminf(bmin[e], ob);
      } else {
        a[e] += oa;
      }
    }
    const bool empty = t_hi <= t_lo;
    const size_t rec = (static_cast<size_t>(phys) * kv.Hkv + h) * g + sub;
    // lanes < 16 write dims 8c..8c+3, lanes >= 16 dims 8c+4..8c+7
    const int e0 = half * 4;
    if (KIND == DSA_META_MINMAX) {
      uint4 o;
      uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float hi = half ? a[4 + e] : a[e];
        const float lo = half ? bmin[4 + e] : bmin[e];
        __nv_bfloat162 pr = __floats2bfloat162_rn(empty ? 0.f : hi, empty ? 0.f : lo);
        w[e] = *reinterpret_cast<uint32_t*>(&pr);
      }
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(meta) + rec * (2 * kHeadDim) +
                           (c * 8 + e0) * 2;
      *reinterpret_cast<uint4*>(dst) = o;
    } else {
      const float cnt = static_cast<float>(max(t_hi - t_lo, 1));
      float4 o;
      o.x = empty ? 0.f : (half ? a[4] : a[0]) / cnt;
      o.y = empty ? 0.f : (half ? a[5] : a[1]) / cnt;
      o.z = empty ? 0.f : (half ? a[6] : a[2]) / cnt;
      o.w = empty ? 0.f : (half ? a[7] : a[3]) / cnt;
      float* dst = reinterpret_cast<float*>(meta) + rec * kHeadDim + c * 8 + e0;
      *reinterpret_cast<float4*>(dst) = o;
    }
  }
}

// One warp per (request, page position, KV head).
template <int KIND>
__global__ void __launch_bounds__(256)
    build_meta_kernel(const KvView kv, const __nv_bfloat16* __restrict__ k_pages, int lp,
                      void* __restrict__ meta) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  const int lane = threadIdx.x & 31;
  const long long item = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int h = static_cast<int>(item % kv.Hkv);
  const long long bj = item / kv.Hkv;
  const int b = static_cast<int>(bj / kv.max_pages), j = static_cast<int>(bj % kv.max_pages);
  if (b >= kv.B) return;
  const int L = request_len(kv, b);
  const int npos = (L + kv.p - 1) / kv.p;
  if (j >= npos) return;
  const int phys = kv.page_table[static_cast<size_t>(b) * kv.max_pages + j];
  if (phys < 0 || phys >= kv.num_phys) {
    if (lane == 0) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
    return;
  }
  page_meta<KIND, false>(kv, k_pages, lp, meta, j, h, phys, L, lane);
}

// One warp per (request, KV head): writes the request's newest token (position L - 1) into its
// page of the pools, then recomputes that page's metadata (when meta is given).
template <int KIND>
__global__ void __launch_bounds__(256)
    append_kv_kernel(const KvView kv, __nv_bfloat16* __restrict__ k_pages,
                     __nv_bfloat16* __restrict__ v_pages, const __nv_bfloat16* __restrict__ k_new,
                     const __nv_bfloat16* __restrict__ v_new, int lp, void* __restrict__ meta) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  const int lane = threadIdx.x & 31;
  const long long item = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int h = static_cast<int>(item % kv.Hkv);
  const int b = static_cast<int>(item / kv.Hkv);
  if (b >= kv.B) return;
  const int L = request_len(kv, b);
  if (L <= 0) return;
  const int t = L - 1, j = t / kv.p;
  const int phys = kv.page_table[static_cast<size_t>(b) * kv.max_pages + j];
  if (phys < 0 || phys >= kv.num_phys) {
    if (lane == 0) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
    return;
  }
  const size_t row = (static_cast<size_t>(phys) * kv.Hkv + h) * kv.p + (t - j * kv.p);
  const size_t src = (static_cast<size_t>(b) * kv.Hkv + h) * kHeadDim;
  const int c = lane & 15;  // lanes 0..15 copy the K row, 16..31 the V row, 16 bytes each
  const __nv_bfloat16* from = (lane < 16 ? k_new : v_new) + src + c * 8;
  __nv_bfloat16* to = (lane < 16 ? k_pages : v_pages) + row * kHeadDim + c * 8;
  *reinterpret_cast<uint4*>(to) = __ldg(reinterpret_cast<const uint4*>(from));
  if (meta == nullptr) return;
  __threadfence_block();
  __syncwarp();  // the new K row is visible to the whole warp
  page_meta<KIND, true>(kv, k_pages, lp, meta, j, h, phys, L, lane);
}

// ------------------------------------------------------------------------------------ scoring
// Record groups of 8 lanes (arithmetic in score_core.cuh).
constexpr int kScoreThreads = 256;
constexpr int kScoreGroups = kScoreThreads / 8;

template <int KIND>
__global__ void __launch_bounds__(kScoreThreads)
    score_kernel(const KvView kv, const __nv_bfloat16* __restrict__ q,
                 const uint8_t* __restrict__ meta, int lp, int pages_per_cta,
                 float* __restrict__ scores, int stride) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  __shared__ float sQbar[kHeadDim];
  const int row = blockIdx.y;
  const int b = row / kv.Hkv, h = row % kv.Hkv;
  const int j0 = blockIdx.x * pages_per_cta;
  const int j1 = min(j0 + pages_per_cta, stride);
  float* out = scores + static_cast<size_t>(row) * stride;
  if (kv.streaming != nullptr && kv.streaming[h] != 0) {
    for (int j = j0 + threadIdx.x; j < j1; j += kScoreThreads) out[j] = -INFINITY;
    return;
  }
  const int g = kv.p / lp;
  const int L = request_len(kv, b);
  const int nl = (L + lp - 1) / lp;
  group_mean_query(q + (static_cast<size_t>(b) * kv.Hq + h * kv.G) * kHeadDim, kv.G, sQbar,
                   threadIdx.x, kScoreThreads);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int gl = lane & 7;
  float qv[16];
  group_query_dims(sQbar, gl, qv);

  const int32_t* table = kv.page_table + static_cast<size_t>(b) * kv.max_pages;
  // warp-uniform loop: warp w, group gi of its 4 groups, handles records jA and jA + 32
  for (int jbase = j0 + (threadIdx.x >> 5) * 4; jbase < j1; jbase += 2 * kScoreGroups) {
    const int jA = jbase + (lane >> 3);
    const int jB = jA + kScoreGroups;
    const bool inA = jA < j1 && jA < nl, inB = jB < j1 && jB < nl;
    const int physA = inA ? table[jA / g] : 0;
    const int physB = inB ? table[jB / g] : 0;
    const bool okA = inA && physA >= 0 && physA < kv.num_phys;
    const bool okB = inB && physB >= 0 && physB < kv.num_phys;
    if (gl == 0 && ((inA && !okA) || (inB && !okB))) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
    uint4 ra[4], rb[4];
    if (okA) load_record(meta, (static_cast<size_t>(physA) * kv.Hkv + h) * g + jA % g, gl, ra);
    if (okB) load_record(meta, (static_cast<size_t>(physB) * kv.Hkv + h) * g + jB % g, gl, rb);
    const float sA = group_sum(okA ? record_partial<KIND>(ra, qv) : 0.f);
    const float sB = group_sum(okB ? record_partial<KIND>(rb, qv) : 0.f);
    if (gl == 0) {
      if (jA < j1) out[jA] = okA ? sA : -INFINITY;
      if (jB < j1) out[jB] = okB ? sB : -INFINITY;
    }
  }
}

}  // namespace

cudaError_t launch_build_meta(const KvView& kv, const __nv_bfloat16* k_pages, int kind, int lp,
                              void* meta, cudaStream_t s) {
  const long long items = static_cast<long long>(kv.B) * kv.max_pages * kv.Hkv;
  const long long blocks = (items + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned nb = static_cast<unsigned>(blocks);
  return kind == DSA_META_MINMAX
             ? launch_pdl(build_meta_kernel<DSA_META_MINMAX>, nb, 256, 0, s, kv, k_pages, lp, meta)
             : launch_pdl(build_meta_kernel<DSA_META_MEAN>, nb, 256, 0, s, kv, k_pages, lp, meta);
}

cudaError_t launch_append_kv(const KvView& kv, __nv_bfloat16* k_pages, __nv_bfloat16* v_pages,
                             const __nv_bfloat16* k_new, const __nv_bfloat16* v_new, int kind,
                             int lp, void* meta, cudaStream_t s) {
  const long long items = static_cast<long long>(kv.B) * kv.Hkv;
  const long long blocks = (items + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned nb = static_cast<unsigned>(blocks);
  return kind == DSA_META_MINMAX
             ? launch_pdl(append_kv_kernel<DSA_META_MINMAX>, nb, 256, 0, s, kv, k_pages, v_pages,
                          k_new, v_new, lp, meta)
             : launch_pdl(append_kv_kernel<DSA_META_MEAN>, nb, 256, 0, s, kv, k_pages, v_pages,
                          k_new, v_new, lp, meta);
}

cudaError_t launch_score(const KvView& kv, const __nv_bfloat16* q, const void* meta, int kind,
                         int lp, float* scores, int stride, cudaStream_t s) {
  const int rows = kv.B * kv.Hkv;
  // Enough CTAs to cover every SM a few times; each group handles 2 records per round.
  int ppc = 2 * kScoreGroups;
  while (ppc > 2 * kScoreGroups / 2 && static_cast<long long>(rows) * ((stride + ppc - 1) / ppc) < 4 * 152)
    ppc /= 2;
  dim3 grid((stride + ppc - 1) / ppc, rows);
  const uint8_t* m = static_cast<const uint8_t*>(meta);
  return kind == DSA_META_MINMAX
             ? launch_pdl(score_kernel<DSA_META_MINMAX>, grid, kScoreThreads, 0, s, kv, q, m, lp,
                          ppc, scores, stride)
             : launch_pdl(score_kernel<DSA_META_MEAN>, grid, kScoreThreads, 0, s, kv, q, m, lp,
                          ppc, scores, stride);
}

}  // namespace dsa
