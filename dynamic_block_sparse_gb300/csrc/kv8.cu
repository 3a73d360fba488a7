// KV8 pages: the KV pool quantised to 8-bit floats (e4m3) with one fp32 scale per (page, KV head,
// token) for K and one for V -- half the bytes of every selected page the attention reads.  The
// quantiser, and split-K attention over KV8 pages on the CUDA cores (lane = token for q.k, lane =
// 4 dims for p.v), whose per-split records the bf16 path's merge combines.
#include <cuda_fp8.h>

#include "attn_core.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr float kE4m3Max = 448.f;  // largest finite e4m3 value
constexpr int kQ8Threads = 256;
constexpr int kQ8Warps = kQ8Threads / 32;

// One warp per (physical page, KV head, token) row of K or V: lane l holds dims 4l .. 4l+3.
__global__ void __launch_bounds__(kQ8Threads)
    quantize_kv8_kernel(const __nv_bfloat16* __restrict__ src, long long n_rows,
                        uint8_t* __restrict__ dst, float* __restrict__ scales) {
  const long long r = static_cast<long long>(blockIdx.x) * kQ8Warps + (threadIdx.x >> 5);
  if (r >= n_rows) return;
  const int lane = threadIdx.x & 31;
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(src + r * kHeadDim) + lane);
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
  float v[4];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[e] = __bfloat162float(x[e]);
    amax = fmaxf(amax, fabsf(v[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // scale: the row's largest magnitude maps to the largest e4m3 value; an all-zero row keeps 0
  const float scale = amax / kE4m3Max;
  uint32_t packed = 0u;
  if (scale > 0.f) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(v[0] / scale, v[1] / scale), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(v[2] / scale, v[3] / scale), __NV_SATFINITE, __NV_E4M3);
    packed = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  reinterpret_cast<uint32_t*>(dst + r * kHeadDim)[lane] = packed;
  if (lane == 0) scales[r] = scale;
}

// Split-K attention over KV8 pages.  CTA (split, row) takes selected pages split, split + splits,
// ... of its row; warp w of it every kQ8Warps-th of those.  A warp keeps the online-softmax state
// (log2 units) of kHeadsPerPass query heads: 32 tokens at a time, lane = token for q.k (its K row
// dequantised as it is read, the row's scale applied to the dot product), then lane = 4 dims for
// p.v (each token's V scale folded into its weight).  Heads beyond kHeadsPerPass take further
// passes over the same pages (L1/L2-resident by then).  Record (split, head): O (normalised),
// m (natural log), l -- the bf16 path's split records.
constexpr int kHeadsPerPass = 4;

DSA_DEV float2 fp8x2_to_float2(uint16_t v) {
  const __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__global__ void __launch_bounds__(kQ8Threads)
    kv8_attn_kernel(const Kv8AttnArgs a) {
  const KvView& kv = a.kv;
  const int split = blockIdx.x, row = blockIdx.y;
  const int b = row / kv.Hkv, h = row % kv.Hkv;
  if (kv.streaming != nullptr && kv.streaming[h] != 0) return;
  const int G = kv.G, page = kv.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float qs[16][kHeadDim];  // the group's queries times scale * log2(e)
  __shared__ float ws_m[kQ8Warps][kHeadsPerPass], ws_l[kQ8Warps][kHeadsPerPass];
  __shared__ __align__(16) float ws_o[kQ8Warps][kHeadsPerPass][kHeadDim];
  for (int e = tid; e < G * kHeadDim; e += kQ8Threads) {
    const int g = e >> 7, d = e & 127;
    const size_t qi = (static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G + g) * kHeadDim;
    qs[g][d] = __bfloat162float(a.q[qi + d]) * a.scale_log2;
  }
  __syncthreads();
  const int L = request_len(kv, b);
  const int npos = (L + page - 1) / page;
  const int cnt = min(max(a.count[row], 0), a.idx_stride);
  const int32_t* sel = a.idx + static_cast<size_t>(row) * a.idx_stride;
  for (int g0 = 0; g0 < G; g0 += kHeadsPerPass) {
    const int ng = min(kHeadsPerPass, G - g0);
    float m[kHeadsPerPass], l[kHeadsPerPass], o[kHeadsPerPass][4];
#pragma unroll
    for (int g = 0; g < kHeadsPerPass; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
      o[g][0] = o[g][1] = o[g][2] = o[g][3] = 0.f;
    }
    for (int i = split + warp * a.splits; i < cnt; i += kQ8Warps * a.splits) {
      const int pos = sel[i];
      int phys = 0;
      if (!lookup_page(kv, b, pos, npos, &phys)) continue;
      const size_t prow = (static_cast<size_t>(phys) * kv.Hkv + h) * page;  // first token row
      for (int c0 = 0; c0 < page; c0 += 32) {
        const int slot = c0 + lane;
        const bool valid = slot < page && pos * page + slot < L;
        // lane = token: its scores for the pass's heads
        float sc[kHeadsPerPass];
#pragma unroll
        for (int g = 0; g < kHeadsPerPass; ++g) sc[g] = -INFINITY;
        if (valid) {
          const uint4* kr = reinterpret_cast<const uint4*>(a.k8 + (prow + slot) * kHeadDim);
          float acc[kHeadsPerPass] = {};
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16 dims per 16-byte piece
            const uint4 raw = __ldg(kr + c);
            const uint16_t* pr = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 kv2 = fp8x2_to_float2(pr[e]);
              const int d = c * 16 + e * 2;
#pragma unroll
              for (int g = 0; g < kHeadsPerPass; ++g) {
                if (g < ng)
                  acc[g] = fmaf(qs[g0 + g][d + 1], kv2.y, fmaf(qs[g0 + g][d], kv2.x, acc[g]));
              }
            }
          }
          const float ksc = __ldg(a.ks + prow + slot);
#pragma unroll
          for (int g = 0; g < kHeadsPerPass; ++g)
            if (g < ng) sc[g] = acc[g] * ksc;
        }
        const float vsc = valid ? __ldg(a.vs + prow + slot) : 0.f;
        // lane = 4 dims: this chunk's V words, then the online-softmax update per head
        uint32_t vw[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int su = c0 + u;
          vw[u] = su < page ? __ldg(reinterpret_cast<const uint32_t*>(a.v8 + (prow + su) * kHeadDim) +
                                    lane)
                            : 0u;
        }
#pragma unroll
        for (int g = 0; g < kHeadsPerPass; ++g) {
          if (g >= ng) break;
          const float cmax = warp_max(sc[g]);
          if (cmax == -INFINITY) continue;
          const float mn = fmaxf(m[g], cmax);
          const float f = m[g] == -INFINITY ? 0.f : fast_exp2(m[g] - mn);
          const float pt = valid ? fast_exp2(sc[g] - mn) : 0.f;
          l[g] = l[g] * f + warp_sum(pt);
          float4 acc = make_float4(o[g][0] * f, o[g][1] * f, o[g][2] * f, o[g][3] * f);
          const float pv = pt * vsc;
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float w = __shfl_sync(0xffffffffu, pv, u);
            if (w == 0.f) continue;  // invalid token (or a zero scale): nothing to add
            const float2 v01 = fp8x2_to_float2(static_cast<uint16_t>(vw[u] & 0xffffu));
            const float2 v23 = fp8x2_to_float2(static_cast<uint16_t>(vw[u] >> 16));
            acc.x = fmaf(w, v01.x, acc.x);
            acc.y = fmaf(w, v01.y, acc.y);
            acc.z = fmaf(w, v23.x, acc.z);
            acc.w = fmaf(w, v23.y, acc.w);
          }
          o[g][0] = acc.x;
          o[g][1] = acc.y;
          o[g][2] = acc.z;
          o[g][3] = acc.w;
          m[g] = mn;
        }
      }
    }
    // the warps' states of the pass's heads -> records
#pragma unroll
    for (int g = 0; g < kHeadsPerPass; ++g) {
      if (g >= ng) break;
      if (lane == 0) {
        ws_m[warp][g] = m[g];
        ws_l[warp][g] = l[g];
      }
      *reinterpret_cast<float4*>(&ws_o[warp][g][lane * 4]) =
          make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
    }
    __syncthreads();
    for (int e = tid; e < ng * kHeadDim; e += kQ8Threads) {
      const int g = e >> 7, d = e & 127;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kQ8Warps; ++w)
        if (ws_l[w][g] > 0.f) M = fmaxf(M, ws_m[w][g]);
      float Ls = 0.f, acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kQ8Warps; ++w) {
          if (!(ws_l[w][g] > 0.f)) continue;
          const float f = fast_exp2(ws_m[w][g] - M);
          Ls += ws_l[w][g] * f;
          acc += ws_o[w][g][d] * f;
        }
      }
      float* rec =
          a.part + ((static_cast<size_t>(row) * a.splits + split) * G + g0 + g) * kRecordFloats;
      rec[d] = Ls > 0.f ? acc / Ls : 0.f;
      if (d == 0) {
        rec[128] = Ls > 0.f ? M * kLn2 : -INFINITY;
        rec[129] = Ls;
      }
    }
    __syncthreads();  // ws_* are rewritten by the next pass
  }
}

}  // namespace

cudaError_t launch_kv8_attn(const Kv8AttnArgs& a, cudaStream_t s) {
  dim3 grid(a.splits, a.kv.B * a.kv.Hkv);
  kv8_attn_kernel<<<grid, kQ8Threads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_kv8(const __nv_bfloat16* src, long long n_rows, uint8_t* dst,
                                float* scales, cudaStream_t s) {
  const long long blocks = (n_rows + kQ8Warps - 1) / kQ8Warps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (blocks == 0) return cudaSuccess;
  quantize_kv8_kernel<<<static_cast<unsigned>(blocks), kQ8Threads, 0, s>>>(src, n_rows, dst,
                                                                           scales);
  return cudaGetLastError();
}

}  // namespace dsa
