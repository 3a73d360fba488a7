// Top-K / hierarchical page selection and the PRR EMA predictor with speculative-set selection.
// One CTA per (request, KV head) row; the row's keys live in shared memory.
#include "internal.h"
#include "score_core.cuh"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kSelectThreads = 512;

// Loads n fp32 values of a row as 16-byte vectors when the row allows it.
template <typename F>
DSA_DEV void for_each_row_value(const float* __restrict__ src, int n, bool vec4, F&& f) {
  if (vec4) {
    for (int j4 = threadIdx.x; j4 * 4 < n; j4 += kSelectThreads) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src) + j4);
      const int j = j4 * 4;
      f(j, v.x);
      if (j + 1 < n) f(j + 1, v.y);
      if (j + 2 < n) f(j + 2, v.z);
      if (j + 3 < n) f(j + 3, v.w);
    }
  } else {
    for (int j = threadIdx.x; j < n; j += kSelectThreads) f(j, __ldg(src + j));
  }
}

__global__ void __launch_bounds__(kSelectThreads)
    select_kernel(const float* __restrict__ scores, int n_logical, int stride, int g, int k,
                  int32_t* __restrict__ idx, int idx_stride, int32_t* __restrict__ count) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  extern __shared__ uint32_t keys[];
  __shared__ SelectAnyScratch<kSelectThreads> sh;
  const int row = blockIdx.x;
  const int n = (n_logical + g - 1) / g;
  const float* s = scores + static_cast<size_t>(row) * stride;
  KeyStats st;
  if (g == 1) {
    const bool vec4 = (stride & 3) == 0 && (reinterpret_cast<uintptr_t>(scores) & 15) == 0;
    for_each_row_value(s, n, vec4, [&](int j, float x) {
      const uint32_t key = score_key(x);
      keys[j] = key;
      st.add(key);
    });
  } else {
    for (int j = threadIdx.x; j < n; j += kSelectThreads) {
      float best = -INFINITY;
      for (int e = 0; e < g; ++e) {
        const int jj = j * g + e;
        if (jj < n_logical) best = fmaxf(best, s[jj]);  // fmaxf drops NaN
      }
      keys[j] = score_key(best);
      st.add(keys[j]);
    }
  }
  __syncthreads();
  int32_t* out = idx + static_cast<size_t>(row) * idx_stride;
  const int total = select_topk_block<kSelectThreads>(keys, n, k, out, sh, st);
  if (threadIdx.x == 0) count[row] = total;
}

__global__ void __launch_bounds__(kSelectThreads)
    ema_kernel(const float* __restrict__ IS, int n, int stride, float* __restrict__ ell,
               float* __restrict__ v, int mode, float alpha, float beta, float gamma,
               float* __restrict__ pred, int k_pred, int32_t* __restrict__ pred_idx,
               int pred_idx_stride, int32_t* __restrict__ pred_count) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  extern __shared__ uint32_t keys[];
  __shared__ SelectAnyScratch<kSelectThreads> sh;
  const int row = blockIdx.x;
  const size_t base = static_cast<size_t>(row) * stride;
  KeyStats st;
  auto update = [&](float is, float l_old, float v_old, float& l_new, float& v_new) {
    ema_step(is, l_old, v_old, mode, alpha, beta, l_new, v_new);
  };
  const bool vec4 = (stride & 3) == 0 && (n & 3) == 0 &&
                    ((reinterpret_cast<uintptr_t>(IS) | reinterpret_cast<uintptr_t>(ell) |
                      reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(pred)) & 15) == 0;
  if (vec4) {
    for (int j4 = threadIdx.x; j4 * 4 < n; j4 += kSelectThreads) {
      const size_t o = base + static_cast<size_t>(j4) * 4;
      const float4 is = __ldg(reinterpret_cast<const float4*>(IS + o));
      float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), vo = lo;
      if (mode != DSA_EMA_INIT) {
        lo = *reinterpret_cast<const float4*>(ell + o);
        vo = *reinterpret_cast<const float4*>(v + o);
      }
      float4 ln, vn, pr;
      update(is.x, lo.x, vo.x, ln.x, vn.x);
      update(is.y, lo.y, vo.y, ln.y, vn.y);
      update(is.z, lo.z, vo.z, ln.z, vn.z);
      update(is.w, lo.w, vo.w, ln.w, vn.w);
      pr.x = ema_predict(ln.x, vn.x, gamma);
      pr.y = ema_predict(ln.y, vn.y, gamma);
      pr.z = ema_predict(ln.z, vn.z, gamma);
      pr.w = ema_predict(ln.w, vn.w, gamma);
      *reinterpret_cast<float4*>(ell + o) = ln;
      *reinterpret_cast<float4*>(v + o) = vn;
      if (pred) *reinterpret_cast<float4*>(pred + o) = pr;
      keys[j4 * 4 + 0] = score_key(pr.x);
      keys[j4 * 4 + 1] = score_key(pr.y);
      keys[j4 * 4 + 2] = score_key(pr.z);
      keys[j4 * 4 + 3] = score_key(pr.w);
      st.add(keys[j4 * 4 + 0]);
      st.add(keys[j4 * 4 + 1]);
      st.add(keys[j4 * 4 + 2]);
      st.add(keys[j4 * 4 + 3]);
    }
  } else {
    for (int j = threadIdx.x; j < n; j += kSelectThreads) {
      float l_new, v_new;
      const float l_old = mode == DSA_EMA_INIT ? 0.f : ell[base + j];
      const float v_old = mode == DSA_EMA_INIT ? 0.f : v[base + j];
      update(IS[base + j], l_old, v_old, l_new, v_new);
      ell[base + j] = l_new;
      v[base + j] = v_new;
      const float p = ema_predict(l_new, v_new, gamma);
      if (pred) pred[base + j] = p;
      keys[j] = score_key(p);
      st.add(keys[j]);
    }
  }
  if (k_pred <= 0 || pred_idx == nullptr) return;
  __syncthreads();
  int32_t* out = pred_idx + static_cast<size_t>(row) * pred_idx_stride;
  const int total = select_topk_block<kSelectThreads>(keys, n, k_pred, out, sh, st);
  if (threadIdx.x == 0) pred_count[row] = total;
}

cudaError_t set_smem(const void* fn, size_t bytes) { return ensure_dynamic_smem(fn, bytes); }

}  // namespace

cudaError_t launch_select(const float* scores, int rows, int n_logical, int stride, int g, int k,
                          int32_t* idx, int idx_stride, int32_t* count, cudaStream_t s) {
  const int n = (n_logical + g - 1) / g;
  const size_t bytes = static_cast<size_t>(n > 0 ? n : 1) * 4;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(select_kernel), bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel, rows, kSelectThreads, bytes, s, scores, n_logical, stride, g, k,
                    idx, idx_stride, count);
}

cudaError_t launch_ema(const float* IS, int rows, int n, int stride, float* ell, float* v,
                       int mode, float alpha, float beta, float gamma, float* pred, int k_pred,
                       int32_t* pred_idx, int pred_idx_stride, int32_t* pred_count,
                       cudaStream_t s) {
  const size_t bytes = static_cast<size_t>(n > 0 ? n : 1) * 4;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(ema_kernel), bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(ema_kernel, rows, kSelectThreads, bytes, s, IS, n, stride, ell, v, mode, alpha,
                    beta, gamma, pred, k_pred, pred_idx, pred_idx_stride, pred_count);
}

}  // namespace dsa
