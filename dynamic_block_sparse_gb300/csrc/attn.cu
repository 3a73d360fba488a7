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
  uint32_t q_off, list_off, bar_off, misc_off, total;
};

__host__ __device__ inline Layout make_layout(int page, int stages) {
  Layout L;
  uint32_t area = 512u * static_cast<uint32_t>(page) * static_cast<uint32_t>(stages);
  if (area < kMergeBytes) area = kMergeBytes;
  area = (area + 1023u) & ~1023u;
  L.q_off = area;
  L.list_off = L.q_off + 16u * kQStride * 2u;
  L.bar_off = L.list_off + kMaxListPages * 8u;
  L.misc_off = L.bar_off + 16u * static_cast<uint32_t>(stages);
  L.total = L.misc_off + 64u + 1024u;  // + slack to align the dynamic base to 1024 bytes
  return L;
}

struct Window {
  int L, sink_end, local_begin;
};

DSA_DEV bool token_in(const Window& w, int t) {
  return t < w.L && (t < w.sink_end || t >= w.local_begin);
}

DSA_DEV bool contains_sorted(const int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int v = a[mid];
    if (v == x) return true;
    if (v < x) lo = mid + 1;
    else hi = mid;
  }
  return false;
}

// Appends the valid candidates of one warp-wide round to the list, preserving order.
DSA_DEV int append_round(bool ok, int phys, int pos, int2* list, int n) {
  const int lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xffffffffu, ok);
  if (ok) {
    const int at = n + __popc(bal & ((1u << lane) - 1u));
    if (at < kMaxListPages) list[at] = make_int2(phys, pos);
  }
  return n + __popc(bal);
}

// Page table lookup of position `pos` of request b, with range checks.
DSA_DEV bool lookup_page(const KvView& kv, int b, int pos, int npos, int* phys) {
  if (pos < 0 || pos >= npos) return false;
  const int ph = kv.page_table[static_cast<size_t>(b) * kv.max_pages + pos];
  if (ph < 0 || ph >= kv.num_phys) {
    raise_status(kv.status, DSA_STATUS_BAD_PAGE);
    return false;
  }
  *phys = ph;
  return true;
}

template <int LIST>
__global__ void __launch_bounds__(kAttnThreads)
    attn_pages_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  const KvView& kv = a.kv;
  const int page = kv.p;
  const int S = a.stages;
  const Layout lay = make_layout(page, S);
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

  if (LIST == LIST_ONE_PAGE) {
    const int cnt = min(max(a.count[row], 0), a.idx_stride);
    if (static_cast<int>(blockIdx.x) >= cnt) return;
  }

  // ---- page list (warp 0)
  if (warp == 0) {
    int n = 0;
    if (LIST == LIST_SELECTED || LIST == LIST_ONE_PAGE) {
      const int cnt = min(max(a.count[row], 0), a.idx_stride);
      int beg, end;
      if (LIST == LIST_ONE_PAGE) {
        beg = blockIdx.x;
        end = beg + 1;
      } else {
        const int chunk = (cnt + a.num_splits - 1) / a.num_splits;
        beg = min(cnt, static_cast<int>(blockIdx.x) * chunk);
        end = min(cnt, beg + chunk);
      }
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
      const int32_t* P = a.spec_idx + static_cast<size_t>(row) * a.spec_stride;
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
        tma_load_2d(dst, &tmK, 0, row0, full);
        tma_load_2d(dst + page * 128, &tmK, 64, row0, full);
        tma_load_2d(dst + 2 * page * 128, &tmV, 0, row0, full);
        tma_load_2d(dst + 3 * page * 128, &tmV, 64, row0, full);
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

// Merges partial records (O, m, l) of one (row, query head) per CTA; thread d owns dim d.
__global__ void __launch_bounds__(128) merge_records_kernel(const MergeArgs a) {
  const int row = blockIdx.x, g = blockIdx.y, d = threadIdx.x;
  const int b = row / a.Hkv, h = row % a.Hkv;
  if (a.streaming != nullptr && a.streaming[h] != 0) return;
  float M = -INFINITY, Lsum = 0.f, acc = 0.f;
  auto fold = [&](const float* rec) {
    const float lp = rec[129];
    if (!(lp > 0.f)) return;
    const float mp = rec[128];
    const float Mn = fmaxf(M, mp);
    const float sa = (M == -INFINITY) ? 0.f : fast_exp2((M - Mn) * kLog2e);
    const float sb = fast_exp2((mp - Mn) * kLog2e) * lp;
    acc = acc * sa + sb * rec[d];
    Lsum = Lsum * sa + sb;
    M = Mn;
  };
  const int nparts = a.count ? min(max(a.count[row], 0), a.slots) : a.slots;
  for (int s = 0; s < nparts; ++s)
    fold(a.part + ((static_cast<size_t>(row) * a.slots + s) * a.G + g) * kRecordFloats);
  if (a.spec_part != nullptr) {
    const int cntP = min(max(a.spec_count[row], 0), a.spec_stride);
    const int cntA = min(max(a.true_count[row], 0), a.true_stride);
    const int32_t* P = a.spec_idx + static_cast<size_t>(row) * a.spec_stride;
    const int32_t* A = a.true_idx + static_cast<size_t>(row) * a.true_stride;
    for (int i = 0; i < cntP; ++i) {
      if (!a.superset && !contains_sorted(A, cntA, P[i])) continue;
      fold(a.spec_part + ((static_cast<size_t>(row) * a.spec_stride + i) * a.G + g) *
                             kRecordFloats);
    }
  }
  const size_t oi = a.out_rows_are_heads
                        ? static_cast<size_t>(b) * a.Hq + static_cast<size_t>(h) * a.G + g
                        : static_cast<size_t>(row) * a.G + g;
  a.out[oi * kHeadDim + d] = Lsum > 0.f ? acc / Lsum : 0.f;
  if (d == 0) {
    a.m[oi] = M;
    a.l[oi] = Lsum;
  }
}

template <int LIST>
cudaError_t launch_list(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a,
                        int grid_x, cudaStream_t s) {
  const Layout lay = make_layout(a.kv.p, a.stages);
  const size_t bytes = lay.total;
  cudaError_t e =
      ensure_dynamic_smem(reinterpret_cast<const void*>(attn_pages_kernel<LIST>), bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(grid_x, a.kv.B * a.kv.Hkv);
  attn_pages_kernel<LIST><<<grid, kAttnThreads, bytes, s>>>(tmK, tmV, a);
  return cudaGetLastError();
}

}  // namespace

size_t attn_smem_bytes(int page, int stages) { return make_layout(page, stages).total; }

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
  dim3 grid(a.rows, a.G);
  merge_records_kernel<<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dsa
