// Top-K / hierarchical page selection and the PRR EMA predictor with speculative-set selection.
// One CTA per (request, KV head) row; the row's keys live in shared memory.
#include "internal.h"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kSelectThreads = 512;

__global__ void __launch_bounds__(kSelectThreads)
    select_kernel(const float* __restrict__ scores, int n_logical, int stride, int g, int k,
                  int32_t* __restrict__ idx, int idx_stride, int32_t* __restrict__ count) {
  extern __shared__ uint32_t keys[];
  __shared__ SelectScratch sh;
  const int row = blockIdx.x;
  const int n = (n_logical + g - 1) / g;
  const float* s = scores + static_cast<size_t>(row) * stride;
  for (int j = threadIdx.x; j < n; j += kSelectThreads) {
    float best = -INFINITY;
    for (int e = 0; e < g; ++e) {
      const int jj = j * g + e;
      if (jj < n_logical) best = fmaxf(best, s[jj]);  // fmaxf drops NaN
    }
    keys[j] = score_key(best);
  }
  __syncthreads();
  const Selection sel = radix_select<kSelectThreads>(keys, n, k, sh);
  int32_t* out = idx + static_cast<size_t>(row) * idx_stride;
  const int total = compact_ascending<kSelectThreads>(keys, n, sel, out, sh);
  for (int i = total + threadIdx.x; i < k; i += kSelectThreads) out[i] = -1;
  if (threadIdx.x == 0) count[row] = total;
}

__global__ void __launch_bounds__(kSelectThreads)
    ema_kernel(const float* __restrict__ IS, int n, int stride, float* __restrict__ ell,
               float* __restrict__ v, int mode, float alpha, float beta, float gamma,
               float* __restrict__ pred, int k_pred, int32_t* __restrict__ pred_idx,
               int pred_idx_stride, int32_t* __restrict__ pred_count) {
  extern __shared__ uint32_t keys[];
  __shared__ SelectScratch sh;
  const int row = blockIdx.x;
  const size_t base = static_cast<size_t>(row) * stride;
  for (int j = threadIdx.x; j < n; j += kSelectThreads) {
    const float is = IS[base + j];
    float l_new = -INFINITY, v_new = 0.f;
    if (is > -INFINITY) {
      const float l_old = ell[base + j];
      if (mode == DSA_EMA_INIT || !(l_old > -INFINITY)) {
        l_new = is;  // no history yet: start from the observed score with zero trend
      } else {
        v_new = beta * (is - l_old) + (1.f - beta) * v[base + j];
        l_new = alpha * is + (1.f - alpha) * l_old;
      }
    }
    ell[base + j] = l_new;
    v[base + j] = v_new;
    const float p = l_new > -INFINITY ? l_new + gamma * v_new : -INFINITY;
    if (pred) pred[base + j] = p;
    keys[j] = score_key(p);
  }
  if (k_pred <= 0 || pred_idx == nullptr) return;
  __syncthreads();
  const Selection sel = radix_select<kSelectThreads>(keys, n, k_pred, sh);
  int32_t* out = pred_idx + static_cast<size_t>(row) * pred_idx_stride;
  const int total = compact_ascending<kSelectThreads>(keys, n, sel, out, sh);
  for (int i = total + threadIdx.x; i < k_pred; i += kSelectThreads) out[i] = -1;
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
  select_kernel<<<rows, kSelectThreads, bytes, s>>>(scores, n_logical, stride, g, k, idx,
                                                    idx_stride, count);
  return cudaGetLastError();
}

cudaError_t launch_ema(const float* IS, int rows, int n, int stride, float* ell, float* v,
                       int mode, float alpha, float beta, float gamma, float* pred, int k_pred,
                       int32_t* pred_idx, int pred_idx_stride, int32_t* pred_count,
                       cudaStream_t s) {
  const size_t bytes = static_cast<size_t>(n > 0 ? n : 1) * 4;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(ema_kernel), bytes);
  if (e != cudaSuccess) return e;
  ema_kernel<<<rows, kSelectThreads, bytes, s>>>(IS, n, stride, ell, v, mode, alpha, beta, gamma,
                                                 pred, k_pred, pred_idx, pred_idx_stride,
                                                 pred_count);
  return cudaGetLastError();
}

}  // namespace dsa
