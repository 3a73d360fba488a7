// Calibration of the PRR EMA predictor (PRR §3.2): for every (alpha, beta, gamma) of the 80-point
// grid, run the predictor over a score trajectory and measure how much of each step's true top-k
// score mass its predicted set covers; the grid point with the largest mean coverage wins.
// One CTA per (row, grid point), the predictor state of its row in shared memory.
#include "internal.h"
#include "score_core.cuh"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kCalibThreads = 512;
constexpr int kCalibWarps = kCalibThreads / 32;
constexpr int kCalibBetas = 5, kCalibGammas = 4;

// Grid point c: alpha outermost (0.2 .. 0.8), then beta (0.1 .. 0.5), gamma innermost
// (0 .. 0.75), the order PRR §3.2's grid is enumerated in.
DSA_DEV void grid_point(int c, float& alpha, float& beta, float& gamma) {
  const int ia = c / (kCalibBetas * kCalibGammas);
  const int ib = (c / kCalibGammas) % kCalibBetas;
  const int ig = c % kCalibGammas;
  alpha = 0.2f * static_cast<float>(ia + 1);
  beta = 0.1f * static_cast<float>(ib + 1);
  gamma = 0.25f * static_cast<float>(ig);
}

// Sum over the CTA (every thread gets it).
DSA_DEV double block_sum(double x, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // red of a previous sum is no longer read
  if (lane == 0) red[warp] = x;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < kCalibWarps; ++w) t += red[w];
  return t;
}

__global__ void __launch_bounds__(kCalibThreads, 1)
    calib_kernel(const float* __restrict__ traj, int T, int rows, int n, int stride, int k,
                 int k_pred, float* __restrict__ H, int32_t* __restrict__ best,
                 unsigned* __restrict__ done) {
  extern __shared__ float cal_smem[];
  float* ell = cal_smem;                                  // [n] level
  float* vt = ell + n;                                    // [n] trend
  uint32_t* keys = reinterpret_cast<uint32_t*>(vt + n);   // [n] ranking keys
  __shared__ SelectAnyScratch<kCalibThreads> sh;
  __shared__ int32_t listP[kMaxListPages], listA[kMaxListPages];  // k, k_pred <= 256
  __shared__ uint32_t bitsP[kCalibMaxN / 32];
  __shared__ double red[kCalibWarps];
  const int tid = threadIdx.x;
  const int row = blockIdx.x / kCalibPoints, c = blockIdx.x % kCalibPoints;
  float alpha, beta, gamma;
  grid_point(c, alpha, beta, gamma);
  const int nwords = (n + 31) >> 5;
  auto step_scores = [&](int t) { return traj + (static_cast<size_t>(t) * rows + row) * stride; };

  {  // the first step initialises the state
    const float* IS = step_scores(0);
    for (int j = tid; j < n; j += kCalibThreads) {
      float l, v;
      ema_step(__ldg(IS + j), 0.f, 0.f, DSA_EMA_INIT, alpha, beta, l, v);
      ell[j] = l;
      vt[j] = v;
    }
  }
  double total = 0.0;
  for (int t = 1; t < T; ++t) {
    const float* IS = step_scores(t);
    // P = the top-k_pred pages of the prediction made before step t's scores are seen
    KeyStats sp;
    __syncthreads();  // keys and lists of the previous step are no longer read
    for (int j = tid; j < n; j += kCalibThreads) {
      keys[j] = score_key(ema_predict(ell[j], vt[j], gamma));
      sp.add(keys[j]);
    }
    for (int w = tid; w < nwords; w += kCalibThreads) bitsP[w] = 0u;
    __syncthreads();
    const int nP = select_topk_block<kCalibThreads>(keys, n, k_pred, listP, sh, sp);
    __syncthreads();
    for (int i = tid; i < nP; i += kCalibThreads) {
      const int j = listP[i];
      atomicOr(&bitsP[j >> 5], 1u << (j & 31));
    }
    // A = the true top-k of step t
    KeyStats sa;
    for (int j = tid; j < n; j += kCalibThreads) {
      keys[j] = score_key(__ldg(IS + j));
      sa.add(keys[j]);
    }
    __syncthreads();
    const int nA = select_topk_block<kCalibThreads>(keys, n, k, listA, sh, sa);
    __syncthreads();
    // the share of A's score mass that P covers (1 when A's scores sum to 0)
    double num = 0.0, den = 0.0;
    for (int i = tid; i < nA; i += kCalibThreads) {
      const int j = listA[i];
      const double s = __ldg(IS + j);
      den += s;
      if ((bitsP[j >> 5] >> (j & 31)) & 1u) num += s;
    }
    num = block_sum(num, red);
    den = block_sum(den, red);
    total += den != 0.0 ? num / den : 1.0;
    // the predictor sees step t's scores
    for (int j = tid; j < n; j += kCalibThreads) {
      float l, v;
      ema_step(__ldg(IS + j), ell[j], vt[j], DSA_EMA_UPDATE, alpha, beta, l, v);
      ell[j] = l;
      vt[j] = v;
    }
  }
  // this grid point's mean coverage; the row's last CTA picks the best (ties to the lower point)
  __shared__ bool last;
  if (tid == 0) {
    H[static_cast<size_t>(row) * kCalibPoints + c] =
        static_cast<float>(total / static_cast<double>(T > 1 ? T - 1 : 1));
    __threadfence();
    last = atomicAdd(done + row, 1u) == static_cast<unsigned>(kCalibPoints - 1);
  }
  __syncthreads();
  if (last && tid < 32) {
    __threadfence();
    float hb = -INFINITY;
    int cb = kCalibPoints;
    for (int i = tid; i < kCalibPoints; i += 32) {
      const float h = __ldcg(H + static_cast<size_t>(row) * kCalibPoints + i);
      if (h > hb) {  // i ascends per lane: the first of equal values stays
        hb = h;
        cb = i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ho = __shfl_xor_sync(0xffffffffu, hb, o);
      const int co = __shfl_xor_sync(0xffffffffu, cb, o);
      if (ho > hb || (ho == hb && co < cb)) {
        hb = ho;
        cb = co;
      }
    }
    if (tid == 0) {
      best[row] = cb < kCalibPoints ? cb : 0;  // no H above -inf: the first point
      done[row] = 0u;                          // left zero for the next call
    }
  }
}

}  // namespace

size_t calib_smem_bytes(int n) { return static_cast<size_t>(n) * 12; }

cudaError_t launch_calib(const float* traj, int T, int rows, int n, int stride, int k, int k_pred,
                         float* H, int32_t* best, unsigned* done, cudaStream_t s) {
  const size_t bytes = calib_smem_bytes(n);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(calib_kernel), bytes);
  if (e != cudaSuccess) return e;
  calib_kernel<<<rows * kCalibPoints, kCalibThreads, bytes, s>>>(traj, T, rows, n, stride, k, k_pred,
                                                                H, best, done);
  return cudaGetLastError();
}

}  // namespace dsa
