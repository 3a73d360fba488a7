// Attention over lists of KV pages: split-K over selected pages, per-page partial records, the
// Lambda window of streaming heads and the repair of missed pages, plus the log-sum-exp merge.
//
// One CTA serves one (request, KV head) row and a slice of its page list, with the whole query
// group of that KV head in one m16 tile, so each selected page crosses HBM once.  Warp 4 is a
// TMA producer feeding a ring of page stages (full/empty mbarriers); warps 0..3 consume 16-token
// tiles round-robin and merge their online-softmax states at the end.
#include "attn_core.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kConsumers = 4;
constexpr int kAttnThreads = (kConsumers + 1) * 32;
constexpr uint32_t kMergeBytes = kConsumers * (16 * 128 + 32) * 4;

struct Layout {
  uint32_t q_off, list_off, bar_off, misc_off, scratch_off, total;
};

// scratch_ints: extra int32 slots (the speculative list of a repair, staged for binary search).
__host__ __device__ inline Layout make_layout(int page, int stages, int scratch_ints) {
  Layout L;
  uint32_t area = 512u * static_cast<uint32_t>(page) * static_cast<uint32_t>(stages);
  if (area < kMergeBytes) area = kMergeBytes;
  area = (area + 1023u) & ~1023u;
  L.q_off = area;
  L.list_off = L.q_off + 16u * kQStride * 2u;
  L.bar_off = L.list_off + kMaxListPages * 8u;
  L.misc_off = L.bar_off + 16u * static_cast<uint32_t>(stages);
  L.scratch_off = L.misc_off + 64u;
  L.total = L.scratch_off + 4u * static_cast<uint32_t>(scratch_ints) + 1024u;  // + align slack
  return L;
}

struct Window {
  int L, sink_end, local_begin;
};

DSA_DEV bool token_in(const Window& w, int t) {
  return t < w.L && (t < w.sink_end || t >= w.local_begin);
}

template <int LIST>
__global__ void __launch_bounds__(kAttnThreads)
    attn_pages_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const KvView& kv = a.kv;
  const int page = kv.p;
  const int S = a.stages;
  const Layout lay = make_layout(page, S, LIST == LIST_REPAIR ? a.spec_stride : 0);
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + lay.q_off);
  int2* list = reinterpret_cast<int2*>(smem + lay.list_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  int* misc = reinterpret_cast<int*>(smem + lay.misc_off);  // [0] n_items, [1] abort
  volatile int* abort_flag = misc + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = blockIdx.y;
  const int b = row / kv.Hkv, h = row % kv.Hkv;
  const bool is_streaming = kv.streaming != nullptr && kv.streaming[h] != 0;
  if ((LIST == LIST_STREAMING) != is_streaming) return;
  const int L = request_len(kv, b);
  const int npos = (L + page - 1) / page;

  Window win;
  win.L = L;
  win.sink_end = 0;
  win.local_begin = 0;
  int out_slot = blockIdx.x;

  int one_pos = -1;
  if (LIST == LIST_ONE_PAGE) {
    // the slot's position and the row's count are independent loads: issue both, then test
    one_pos = a.idx[static_cast<size_t>(row) * a.idx_stride + blockIdx.x];
    const int cnt = min(max(a.count[row], 0), a.idx_stride);
    if (static_cast<int>(blockIdx.x) >= cnt) return;
  }
  int32_t* sP = reinterpret_cast<int32_t*>(smem + lay.scratch_off);
  if (LIST == LIST_REPAIR) {
    const int cntP = min(max(a.spec_count[row], 0), a.spec_stride);
    const int32_t* P = a.spec_idx + static_cast<size_t>(row) * a.spec_stride;
    for (int i = tid; i < cntP; i += kAttnThreads) sP[i] = P[i];
    __syncthreads();
  }

  // ---- page list (warp 0)
  if (warp == 0) {
    int n = 0;
    if (LIST == LIST_ONE_PAGE) {
      int phys = 0;
      const bool ok = lane == 0 && lookup_page(kv, b, one_pos, npos, &phys);
      n = append_round(ok, phys, one_pos, list, n);
    } else if (LIST == LIST_SELECTED) {
      const int cnt = min(max(a.count[row], 0), a.idx_stride);
      const int chunk = (cnt + a.num_splits - 1) / a.num_splits;
      const int beg = min(cnt, static_cast<int>(blockIdx.x) * chunk);
      const int end = min(cnt, beg + chunk);
      const int32_t* sel = a.idx + static_cast<size_t>(row) * a.idx_stride;
      for (int base = beg; base < end; base += 32) {
        const int i = base + lane;
        int phys = 0, pos = -1;
        bool ok = false;
        if (i < end) {
          pos = sel[i];
          ok = lookup_page(kv, b, pos, npos, &phys);
        }
        n = append_round(ok, phys, pos, list, n);
      }
    } else if (LIST == LIST_STREAMING) {
      win.sink_end = min(a.sink, L);
      win.local_begin = max(0, L - a.local);
      const int first_end = (win.sink_end + page - 1) / page;
      const int second_beg = max(first_end, win.local_begin / page);
      const int n_first = first_end;
      const int n_total = n_first + max(0, npos - second_beg);
      for (int base = 0; base < n_total; base += 32) {
        const int i = base + lane;
        int phys = 0, pos = -1;
        bool ok = false;
        if (i < n_total) {
          pos = i < n_first ? i : second_beg + (i - n_first);
          ok = lookup_page(kv, b, pos, npos, &phys);
        }
        n = append_round(ok, phys, pos, list, n);
      }
    } else {  // LIST_REPAIR: missed pages A \ P, this split's share
      const int cntA = min(max(a.count[row], 0), a.idx_stride);
      const int cntP = min(max(a.spec_count[row], 0), a.spec_stride);
      const int32_t* A = a.idx + static_cast<size_t>(row) * a.idx_stride;
      const int32_t* P = sP;
      int missed_total = 0;
      for (int base = 0; base < cntA; base += 32) {
        const int i = base + lane;
        const bool miss = i < cntA && !contains_sorted(P, cntP, A[i]);
        missed_total += __popc(__ballot_sync(0xffffffffu, miss));
      }
      const int chunk = (missed_total + a.num_splits - 1) / a.num_splits;
      const int beg = min(missed_total, static_cast<int>(blockIdx.x) * chunk);
      const int end = min(missed_total, beg + chunk);
      int rank = 0;
      for (int base = 0; base < cntA && rank < end; base += 32) {
        const int i = base + lane;
        const bool miss = i < cntA && !contains_sorted(P, cntP, A[i]);
        const unsigned bal = __ballot_sync(0xffffffffu, miss);
        const int my_rank = rank + __popc(bal & ((1u << lane) - 1u));
        int phys = 0, pos = -1;
        bool ok = false;
        if (miss && my_rank >= beg && my_rank < end) {
          pos = A[i];
          ok = lookup_page(kv, b, pos, npos, &phys);
        }
        n = append_round(ok, phys, pos, list, n);
        rank += __popc(bal);
      }
    }
    if (lane == 0) {
      misc[0] = min(n, kMaxListPages);
      misc[1] = 0;
    }
  }
  if (LIST == LIST_STREAMING) {
    win.sink_end = min(a.sink, L);
    win.local_begin = max(0, L - a.local);
  }

  // ---- stage the query group (rows >= G are zero)
  for (int e = tid; e < 16 * 16; e += kAttnThreads) {
    const int r = e >> 4, c = e & 15;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < kv.G)
      v = *reinterpret_cast<const uint4*>(
          a.q + (static_cast<size_t>(b) * kv.Hq + h * kv.G + r) * kHeadDim + c * 8);
    *reinterpret_cast<uint4*>(sQ + r * kQStride + c * 8) = v;
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[S + s]), kConsumers);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int n_items = misc[0];
  const uint32_t stage_bytes = 512u * page;
  const uint32_t smem_base = smem_u32(smem);

  WarpSoftmaxState st;
  state_init(st);

  if (warp == kConsumers) {
    // ---- producer
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      for (int i = 0; i < n_items; ++i) {
        const int s = i % S, u = i / S;
        if (u > 0 && !mbar_wait(smem_u32(&bars[S + s]), (u - 1) & 1, abort_flag, kv.status))
          break;
        const uint32_t full = smem_u32(&bars[s]);
        const uint32_t dst = smem_base + s * stage_bytes;
        const int row0 = (list[i].x * kv.Hkv + h) * page;
        mbar_arrive_expect_tx(full, stage_bytes);
        tma_load_page(dst, &tmK, row0, full);
        tma_load_page(dst + 2 * page * 128, &tmV, row0, full);
      }
    }
  } else {
    // ---- consumers
    uint32_t qa[8][4];
    load_q_frags(sQ, qa);
    const int tiles = page / 16;
    int gkt = 0;
    for (int i = 0; i < n_items; ++i) {
      const int s = i % S, u = i / S;
      if (!mbar_wait(smem_u32(&bars[s]), u & 1, abort_flag, kv.status)) break;
      const int pos = list[i].y;
      const uint32_t kb = smem_base + s * stage_bytes;
      const uint32_t vb = kb + 2 * page * 128;
      bool wrote = false;
      for (int t = 0; t < tiles; ++t) {
        if (((gkt + t) & (kConsumers - 1)) != warp) continue;
        const int tok0 = pos * page + t * 16;
        const bool in = token_in(win, tok0 + (lane & 15));
        const uint32_t valid = __ballot_sync(0xffffffffu, in) & 0xffffu;
        if (valid == 0u) continue;
        if (valid != 0xffffu)
          wrote |= zero_invalid_v_rows(valid, smem + s * stage_bytes + 2 * page * 128, page,
                                       t * 16);
        float sc[2][4];
        tile_scores(qa, kb, page, t * 16, sc);
        tile_softmax_pv(st, sc, a.scale_log2, valid, vb, page, t * 16);
      }
      gkt += tiles;
      if (wrote) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[S + s]));
    }
    state_finish(st);
  }
  __syncthreads();
  if (*abort_flag) return;

  // ---- merge the consumer warps' states
  float* sO = reinterpret_cast<float*>(smem);
  float* sM = sO + kConsumers * 2048;
  float* sL = sM + kConsumers * 16;
  if (warp < kConsumers) state_store(st, sO + warp * 2048, sM + warp * 16, sL + warp * 16);
  __syncthreads();

  const bool final_out =
      (LIST == LIST_STREAMING) || (LIST == LIST_SELECTED && a.num_splits == 1);
  if (!final_out && n_items == 0) {  // an empty part: the merge reads only its (m, l)
    for (int g = tid; g < kv.G; g += kAttnThreads) {
      float* rec = a.part +
                   ((static_cast<size_t>(row) * a.part_slots + out_slot) * kv.G + g) * kRecordFloats;
      *reinterpret_cast<float4*>(rec + 128) = make_float4(-INFINITY, 0.f, 0.f, 0.f);
    }
    return;
  }
  for (int e = tid; e < kv.G * kHeadDim; e += kAttnThreads) {
    const int g = e >> 7, d = e & 127;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, sM[w * 16 + g]);
    float Lsum = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float mw = sM[w * 16 + g];
        if (mw == -INFINITY) continue;
        const float f = fast_exp2(mw - M);
        Lsum += sL[w * 16 + g] * f;
        acc += sO[w * 2048 + g * 128 + d] * f;
      }
    }
    const float O = Lsum > 0.f ? acc / Lsum : 0.f;
    const float m_nat = M == -INFINITY ? -INFINITY : M * kLn2;
    if (final_out) {
      const size_t qh = static_cast<size_t>(b) * kv.Hq + h * kv.G + g;
      a.out[qh * kHeadDim + d] = O;
      if (d == 0) {
        a.m[qh] = m_nat;
        a.l[qh] = Lsum;
      }
    } else {
      float* rec = a.part +
                   ((static_cast<size_t>(row) * a.part_slots + out_slot) * kv.G + g) * kRecordFloats;
      rec[d] = O;
      if (d == 0) {
        rec[128] = m_nat;
        rec[129] = Lsum;
        rec[130] = 0.f;
        rec[131] = 0.f;
      }
    }
  }
}

// Merges partial records (O, m, l) of one (row, query head) per CTA.  The parts (split records,
// plus the speculative records of hit pages for a repair) are listed in shared memory, their
// weights l * exp(m - M) computed in parallel, and the weighted sum of the O vectors is split
// over 8 warps (each lane owns 4 dimensions) so that many independent loads are in flight.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

struct MergeLayout {
  size_t w_off, a_off, acc_off, total;
};

// Shared-memory layout of the merge: record pointers, weights, the true set, per-warp partial
// sums; every region starts on a 16-byte boundary (the partial sums are written as float4).
__host__ __device__ inline MergeLayout merge_layout(int max_parts, int a_ints) {
  auto up16 = [](size_t x) { return (x + 15) & ~static_cast<size_t>(15); };
  MergeLayout L;
  L.w_off = up16(static_cast<size_t>(max_parts) * sizeof(const float*));
  L.a_off = up16(L.w_off + static_cast<size_t>(max_parts) * sizeof(float));
  L.acc_off = up16(L.a_off + static_cast<size_t>(a_ints) * sizeof(int32_t));
  L.total = L.acc_off + static_cast<size_t>(kMergeWarps) * 128 * sizeof(float);
  return L;
}

__global__ void __launch_bounds__(kMergeThreads) merge_records_kernel(const MergeArgs a) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  extern __shared__ __align__(16) uint8_t msm[];
  const int row = blockIdx.x, g = blockIdx.y;
  const int b = row / a.Hkv, h = row % a.Hkv;
  if (a.streaming != nullptr && a.streaming[h] != 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int max_parts = a.slots + (a.spec_part != nullptr ? a.spec_stride : 0);
  const MergeLayout lay = merge_layout(max_parts, a.spec_part != nullptr ? a.true_stride : 0);
  const float** s_rec = reinterpret_cast<const float**>(msm);
  float* s_w = reinterpret_cast<float*>(msm + lay.w_off);
  int32_t* s_A = reinterpret_cast<int32_t*>(msm + lay.a_off);
  float* s_acc = reinterpret_cast<float*>(msm + lay.acc_off);
  __shared__ int s_red[33];
  __shared__ float s_f[33];

  const int nsplit = a.count ? min(max(a.count[row], 0), a.slots) : a.slots;
  for (int s = tid; s < nsplit; s += kMergeThreads)
    s_rec[s] = a.part + ((static_cast<size_t>(row) * a.slots + s) * a.G + g) * kRecordFloats;
  int nparts = nsplit;
  if (a.spec_part != nullptr) {
    const int cntP = min(max(a.spec_count[row], 0), a.spec_stride);
    const int cntA = min(max(a.true_count[row], 0), a.true_stride);
    const int32_t* P = a.spec_idx + static_cast<size_t>(row) * a.spec_stride;
    const int32_t* A = a.true_idx + static_cast<size_t>(row) * a.true_stride;
    for (int i = tid; i < cntA; i += kMergeThreads) s_A[i] = A[i];
    __syncthreads();
    // hits in index order, one block-wide round per kMergeThreads entries of P
    for (int base = 0; base < cntP; base += kMergeThreads) {
      const int i = base + tid;
      const bool hit = i < cntP && (a.superset || contains_sorted(s_A, cntA, P[i]));
      int total;
      const int at = block_exclusive_scan(hit ? 1 : 0, s_red, &total);
      if (hit)
        s_rec[nparts + at] = a.spec_part +
                             ((static_cast<size_t>(row) * a.spec_stride + i) * a.G + g) * kRecordFloats;
      nparts += total;
    }
  }
  __syncthreads();
  // weights: M = max m over non-empty parts, w = l exp(m - M), L = sum w
  float mloc = -INFINITY;
  for (int k = tid; k < nparts; k += kMergeThreads) {
    const float* r = s_rec[k];
    const float lp = r[129], mp = r[128];
    s_w[k] = lp;
    if (lp > 0.f) mloc = fmaxf(mloc, mp);
  }
  mloc = warp_max(mloc);
  if (lane == 0) s_f[warp] = mloc;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, s_f[w]);
  __syncthreads();
  float lsum = 0.f;
  for (int k = tid; k < nparts; k += kMergeThreads) {
    const float lp = s_w[k];
    const float wk = lp > 0.f ? lp * fast_exp2((s_rec[k][128] - M) * kLog2e) : 0.f;
    s_w[k] = wk;
    lsum += wk;
  }
  lsum = warp_sum(lsum);
  if (lane == 0) s_f[warp] = lsum;
  __syncthreads();
  float Lsum = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Lsum += s_f[w];
  // weighted sum of O: warp w takes parts w, w + 8, ...; lane owns dims 4*lane .. 4*lane + 3
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int k = warp;
  for (; k + 3 * kMergeWarps < nparts; k += 4 * kMergeWarps) {
    float4 v[4];
    float wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      wv[u] = s_w[k + u * kMergeWarps];  // empty parts (weight 0) are never read
      v[u] = wv[u] > 0.f ? *reinterpret_cast<const float4*>(s_rec[k + u * kMergeWarps] + lane * 4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc.x += wv[u] * v[u].x;
      acc.y += wv[u] * v[u].y;
      acc.z += wv[u] * v[u].z;
      acc.w += wv[u] * v[u].w;
    }
  }
  for (; k < nparts; k += kMergeWarps) {
    const float wk = s_w[k];
    if (!(wk > 0.f)) continue;
    const float4 v = *reinterpret_cast<const float4*>(s_rec[k] + lane * 4);
    acc.x += wk * v.x;
    acc.y += wk * v.y;
    acc.z += wk * v.z;
    acc.w += wk * v.w;
  }
  *reinterpret_cast<float4*>(s_acc + warp * 128 + lane * 4) = acc;
  __syncthreads();
  const size_t oi = a.out_rows_are_heads
                        ? static_cast<size_t>(b) * a.Hq + static_cast<size_t>(h) * a.G + g
                        : static_cast<size_t>(row) * a.G + g;
  if (tid < kHeadDim) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) o += s_acc[w * 128 + tid];
    a.out[oi * kHeadDim + tid] = Lsum > 0.f ? o / Lsum : 0.f;
  }
  if (tid == 0) {
    a.m[oi] = Lsum > 0.f ? M : -INFINITY;
    a.l[oi] = Lsum;
  }
}

template <int LIST>
cudaError_t launch_list(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a,
                        int grid_x, cudaStream_t s) {
  constexpr int list = LIST;
  const Layout lay = make_layout(a.kv.p, a.stages, list == LIST_REPAIR ? a.spec_stride : 0);
  const size_t bytes = lay.total;
  cudaError_t e =
      ensure_dynamic_smem(reinterpret_cast<const void*>(attn_pages_kernel<LIST>), bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(grid_x, a.kv.B * a.kv.Hkv);
  return launch_pdl(attn_pages_kernel<LIST>, grid, kAttnThreads, bytes, s, tmK, tmV, a);
}

}  // namespace

size_t attn_smem_bytes(int page, int stages, int scratch_ints) {
  return make_layout(page, stages, scratch_ints).total;
}

cudaError_t launch_attn(int list, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const AttnArgs& a, int grid_x, cudaStream_t s) {
  switch (list) {
    case LIST_SELECTED: return launch_list<LIST_SELECTED>(tmK, tmV, a, grid_x, s);
    case LIST_ONE_PAGE: return launch_list<LIST_ONE_PAGE>(tmK, tmV, a, grid_x, s);
    case LIST_STREAMING: return launch_list<LIST_STREAMING>(tmK, tmV, a, grid_x, s);
    case LIST_REPAIR: return launch_list<LIST_REPAIR>(tmK, tmV, a, grid_x, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s) {
  const size_t bytes =
      merge_layout(a.slots + (a.spec_part ? a.spec_stride : 0), a.spec_part ? a.true_stride : 0)
          .total;
  if (bytes > 200 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(merge_records_kernel), bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.rows, a.G);
  return launch_pdl(merge_records_kernel, grid, kMergeThreads, bytes, s, a);
}

}  // namespace dsa
