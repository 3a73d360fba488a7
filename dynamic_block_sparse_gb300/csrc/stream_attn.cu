// Persistent split-K sparse attention over many rows: one launch, one CTA per SM.
//
// Every dense (request, KV head) row's selected pages are cut into the same number of chunks, as
// many as keep one (row, chunk) unit per CTA of the grid.  In each CTA warp 8 is a TMA producer:
// it resolves the unit's page-table entries 32 at a time and streams the K/V pages through a
// 128 KB ring, publishing each stage's page position in shared memory; warps 0..7 attend with the
// mma core (eight consumer warps per SM keep enough 16-token tiles in flight to cover the mma
// latency).  At the end of a unit the consumers merge their states, write the unit's partial
// record (O, m, l per query head) to the workspace and take a ticket on the row's counter; the CTA
// that takes the last ticket merges the row's records in chunk order (deterministic) and writes
// the final rows.
#include "attn_core.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kSW = 8;                     // consumer warps
constexpr int kSThreads = (kSW + 1) * 32;  // + one TMA producer warp
constexpr int kSConsumers = kSW * 32;
constexpr uint32_t kSMergeBytes = kSW * (16 * 128 + 32) * 4;
constexpr int kSMaxHeads = 1024;           // KV heads the dense-head table can hold

struct SLayout {
  uint32_t merge_off, q_off, bar_off, misc_off, total;
};

__host__ __device__ inline SLayout slayout(int page, int stages) {
  SLayout L;
  L.merge_off = ((512u * page * stages) + 1023u) & ~1023u;
  L.q_off = L.merge_off + kSMergeBytes;
  L.bar_off = L.q_off + 16u * kQStride * 2u;
  L.misc_off = L.bar_off + 16u * static_cast<uint32_t>(stages);
  L.total = L.misc_off + 256u + 4u * kSMaxHeads + 1024u;
  return L;
}

__global__ void __launch_bounds__(kSThreads, 1)
    stream_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const StreamAttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  const KvView& kv = a.kv;
  const int page = kv.p;
  const int S = a.stages;
  const int G = kv.G;
  const SLayout lay = slayout(page, S);
  float* sO = reinterpret_cast<float*>(smem + lay.merge_off);
  float* sM = sO + kSW * 2048;
  float* sL = sM + kSW * 16;
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + lay.q_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bar_off);  // [S] full, [S] empty
  int* misc = reinterpret_cast<int*>(smem + lay.misc_off);
  volatile int* abort_flag = misc;          // [0]
  volatile int* last_flag = misc + 1;       // [1]
  volatile int* stage_ok = misc + 16;       // [16, 32): did the producer load this stage
  volatile int* stage_pos = misc + 32;      // [32, 48): page position held by this stage
  int* dense_heads = misc + 64;             // [64, 64 + Hkv)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t stage_bytes = 512u * page;
  const uint32_t smem_base = smem_u32(smem);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[S + s]), kSW);
    }
    fence_mbar_init();
    misc[0] = 0;
    int nd = 0;
    for (int hh = 0; hh < kv.Hkv; ++hh)
      if (kv.streaming == nullptr || kv.streaming[hh] == 0) dense_heads[nd++] = hh;
    misc[2] = nd;
  }
  __syncthreads();
  const int nd_heads = misc[2];
  const int n_dense = kv.B * nd_heads;
  int chunks = n_dense > 0 ? static_cast<int>(gridDim.x) / n_dense : 1;
  chunks = max(1, min(chunks, a.chunks));
  const int chunk_pages = (a.idx_stride + chunks - 1) / chunks;
  const int units_total = n_dense * chunks;

  // unit u -> (row, selected slots [beg, end))
  auto unit_range = [&](int u, int* row, int* beg, int* end) {
    const int di = u / chunks;
    const int c = u - di * chunks;
    *row = (di / nd_heads) * kv.Hkv + dense_heads[di % nd_heads];
    const int cnt = min(max(a.count[*row], 0), a.idx_stride);
    *beg = min(cnt, c * chunk_pages);
    *end = min(cnt, *beg + chunk_pages);
  };

  if (warp == kSW) {
    // ---- producer
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
    }
    int i = 0;  // ring position
    for (int u = blockIdx.x; u < units_total && !*abort_flag; u += gridDim.x) {
      int row, beg, end;
      unit_range(u, &row, &beg, &end);
      const int b = row / kv.Hkv, h = row % kv.Hkv;
      const int npos = (request_len(kv, b) + page - 1) / page;
      const int32_t* sel = a.idx + static_cast<size_t>(row) * a.idx_stride;
      bool stopped = false;
      for (int base = beg; base < end && !stopped; base += 32) {
        const int j = base + lane;
        int pos = -1, phys = 0;
        bool ok = false;
        if (j < end) {
          pos = sel[j];
          ok = lookup_page(kv, b, pos, npos, &phys);
        }
        const int nb = min(32, end - base);
        for (int k = 0; k < nb; ++k, ++i) {
          const int pk = __shfl_sync(0xffffffffu, pos, k);
          const int phk = __shfl_sync(0xffffffffu, phys, k);
          const int okk = __shfl_sync(0xffffffffu, ok ? 1 : 0, k);
          const int s = i % S, uu = i / S;
          int stop = 0;
          if (lane == 0 && uu > 0 &&
              !mbar_wait(smem_u32(&bars[S + s]), (uu - 1) & 1, abort_flag, kv.status))
            stop = 1;
          if (__shfl_sync(0xffffffffu, stop, 0)) {  // the whole warp leaves together
            stopped = true;
            break;
          }
          if (lane == 0) {
            const uint32_t full = smem_u32(&bars[s]);
            stage_pos[s] = pk;
            stage_ok[s] = okk;  // both published by the arrive below
            if (!okk) {
              mbar_arrive(full);  // nothing to load: complete the phase with a plain arrival
            } else {
              const uint32_t dst = smem_base + s * stage_bytes;
              const int row0 = (phk * kv.Hkv + h) * page;
              mbar_arrive_expect_tx(full, stage_bytes);
              tma_load_2d(dst, &tmK, 0, row0, full);
              tma_load_2d(dst + page * 128, &tmK, 64, row0, full);
              tma_load_2d(dst + 2 * page * 128, &tmV, 0, row0, full);
              tma_load_2d(dst + 3 * page * 128, &tmV, 64, row0, full);
            }
          }
        }
      }
    }
    return;  // the producer takes no part in the epilogues (they use named barrier 1)
  }

  // ---- consumers
  const int tiles = page / 16;
  int i = 0;  // ring position, in lock-step with the producer
  for (int u = blockIdx.x; u < units_total; u += gridDim.x) {
    int row, beg, end;
    unit_range(u, &row, &beg, &end);
    const int b = row / kv.Hkv, h = row % kv.Hkv;
    const int L = request_len(kv, b);
    named_barrier(1, kSConsumers);
    for (int e = tid; e < 16 * 16; e += kSConsumers) {
      const int r = e >> 4, c = e & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < G)
        v = *reinterpret_cast<const uint4*>(
            a.q + (static_cast<size_t>(b) * kv.Hq + h * G + r) * kHeadDim + c * 8);
      *reinterpret_cast<uint4*>(sQ + r * kQStride + c * 8) = v;
    }
    named_barrier(1, kSConsumers);
    uint32_t qa[8][4];
    load_q_frags(sQ, qa);
    WarpSoftmaxState st;
    state_init(st);
    int gkt = 0;
    for (int j = beg; j < end; ++j, ++i) {
      const int s = i % S, uu = i / S;
      if (!mbar_wait(smem_u32(&bars[s]), uu & 1, abort_flag, kv.status)) break;
      const int pos = stage_pos[s];
      const bool loaded = stage_ok[s] != 0;
      const uint32_t kb = smem_base + s * stage_bytes;
      const uint32_t vb = kb + 2 * page * 128;
      bool wrote = false;
      for (int t = 0; loaded && t < tiles; ++t) {
        if (((gkt + t) & (kSW - 1)) != warp) continue;
        const bool in = pos * page + t * 16 + (lane & 15) < L;
        const uint32_t vm = __ballot_sync(0xffffffffu, in) & 0xffffu;
        if (vm == 0u) continue;
        if (vm != 0xffffu)
          wrote |= zero_invalid_v_rows(vm, smem + s * stage_bytes + 2 * page * 128, page, t * 16);
        float sc[2][4];
        tile_scores(qa, kb, page, t * 16, sc);
        tile_softmax_pv(st, sc, a.scale_log2, vm, vb, page, t * 16);
      }
      gkt += tiles;
      if (wrote) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[S + s]));
    }
    state_finish(st);

    // ---- unit epilogue: merge the warps, write the unit's record, take a ticket
    state_store(st, sO + warp * 2048, sM + warp * 16, sL + warp * 16);
    named_barrier(1, kSConsumers);
    const int c = u % chunks;
    float* rec0 = a.part + (static_cast<size_t>(row) * a.chunks + c) * G * kRecordFloats;
    for (int e = tid; e < G * kHeadDim; e += kSConsumers) {
      const int g = e >> 7, d = e & 127;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kSW; ++w) M = fmaxf(M, sM[w * 16 + g]);
      float Lsum = 0.f, acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kSW; ++w) {
          const float mw = sM[w * 16 + g];
          if (mw == -INFINITY) continue;
          const float f = fast_exp2(mw - M);
          Lsum += sL[w * 16 + g] * f;
          acc += sO[w * 2048 + g * 128 + d] * f;
        }
      }
      float* rec = rec0 + g * kRecordFloats;
      rec[d] = Lsum > 0.f ? acc / Lsum : 0.f;
      if (d == 0) {
        rec[128] = Lsum > 0.f ? M * kLn2 : -INFINITY;
        rec[129] = Lsum;
      }
    }
    __threadfence();
    named_barrier(1, kSConsumers);
    if (tid == 0) *last_flag = atomicAdd(a.counters + row, 1) == chunks - 1;
    named_barrier(1, kSConsumers);
    if (*last_flag) {
      // last unit of this row: merge its chunk records in chunk order.  The merge area is free
      // again and holds each record's m and weight and each head's (M, L).
      __threadfence();
      const int C = chunks;
      const float* base = a.part + static_cast<size_t>(row) * a.chunks * G * kRecordFloats;
      float* s_m = sO;            // [G][C]
      float* s_w = sO + G * C;    // [G][C]
      float* s_ml = s_w + G * C;  // [G][2]
      for (int e = tid; e < G * C; e += kSConsumers) {
        const int g = e / C, cc = e - g * C;
        const float* r = base + (static_cast<size_t>(cc) * G + g) * kRecordFloats;
        s_m[e] = __ldcg(r + 128);
        s_w[e] = __ldcg(r + 129);
      }
      named_barrier(1, kSConsumers);
      for (int g = warp; g < G; g += kSW) {
        float M = -INFINITY;
        for (int cc = lane; cc < C; cc += 32)
          if (s_w[g * C + cc] > 0.f) M = fmaxf(M, s_m[g * C + cc]);
        M = warp_max(M);
        float Ls = 0.f;
        for (int cc = lane; cc < C; cc += 32) {
          const float lp = s_w[g * C + cc];
          const float wgt = lp > 0.f ? lp * fast_exp2((s_m[g * C + cc] - M) * kLog2e) : 0.f;
          s_w[g * C + cc] = wgt;
          Ls += wgt;
        }
        Ls = warp_sum(Ls);
        if (lane == 0) {
          s_ml[2 * g] = M;
          s_ml[2 * g + 1] = Ls;
        }
      }
      named_barrier(1, kSConsumers);
      // warp w finalises heads w, w + 8, ...; lane owns dims 4*lane .. 4*lane + 3
      for (int g = warp; g < G; g += kSW) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int cc = 0;
        for (; cc + 8 <= C; cc += 8) {
          float4 v[8];
          float wv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            wv[k] = s_w[g * C + cc + k];
            v[k] = wv[k] > 0.f
                       ? __ldcg(reinterpret_cast<const float4*>(
                                    base + (static_cast<size_t>(cc + k) * G + g) * kRecordFloats) +
                                lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            acc.x += wv[k] * v[k].x;
            acc.y += wv[k] * v[k].y;
            acc.z += wv[k] * v[k].z;
            acc.w += wv[k] * v[k].w;
          }
        }
        for (; cc < C; ++cc) {
          const float wk = s_w[g * C + cc];
          if (!(wk > 0.f)) continue;
          const float4 v = __ldcg(
              reinterpret_cast<const float4*>(base + (static_cast<size_t>(cc) * G + g) *
                                                         kRecordFloats) +
              lane);
          acc.x += wk * v.x;
          acc.y += wk * v.y;
          acc.z += wk * v.z;
          acc.w += wk * v.w;
        }
        const float Ls = s_ml[2 * g + 1];
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const size_t qh = static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G + g;
        *reinterpret_cast<float4*>(a.out + qh * kHeadDim + lane * 4) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (lane == 0) {
          a.m[qh] = Ls > 0.f ? s_ml[2 * g] : -INFINITY;
          a.l[qh] = Ls;
        }
      }
      if (tid == 0) a.counters[row] = 0;  // ready for the next call
    }
  }
}

}  // namespace

size_t stream_attn_smem_bytes(int page, int stages) { return slayout(page, stages).total; }

cudaError_t launch_stream_attn(const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const StreamAttnArgs& a, cudaStream_t s) {
  const size_t bytes = slayout(a.kv.p, a.stages).total;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(stream_attn_kernel), bytes);
  if (e != cudaSuccess) return e;
  // a persistent grid: as many CTAs as are resident at once
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_attn_kernel, kSThreads,
                                                         bytes)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  stream_attn_kernel<<<per_sm * sms, kSThreads, bytes, s>>>(tmK, tmV, a);
  return cudaGetLastError();
}

}  // namespace dsa
