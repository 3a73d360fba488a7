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

// The predictor state of a CTA lives in the workspace (L2-resident; its row's level and trend of
// this grid point), the ranking keys in shared memory, so that several CTAs share an SM and the
// whole grid of (row, point) CTAs runs in one wave.  A_t of every (row, step) was selected once
// beforehand (it does not depend on the grid point).
__global__ void __launch_bounds__(kCalibThreads, 2)
    calib_kernel(const float* __restrict__ traj, int T, int rows, int n, int stride, int k,
                 int k_pred, const int32_t* __restrict__ a_idx, const int32_t* __restrict__ a_cnt,
                 float* __restrict__ state, float* __restrict__ H, int32_t* __restrict__ best,
                 unsigned* __restrict__ done) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  extern __shared__ uint32_t keys[];  // [n] ranking keys of the prediction
  __shared__ SelectAnyScratch<kCalibThreads> sh;
  __shared__ int32_t listP[kMaxListPages];  // k_pred <= 256
  __shared__ uint32_t bitsP[kCalibMaxN / 32];
  __shared__ unsigned s_bound;
  __shared__ int s_nc;
  TopkScratch& ts = sh.small;
  const int tid = threadIdx.x, lane = tid & 31;
  const int row = blockIdx.x / kCalibPoints, c = blockIdx.x % kCalibPoints;
  float alpha, beta, gamma;
  grid_point(c, alpha, beta, gamma);
  const int nwords = (n + 31) >> 5;
  float* ell = state + static_cast<size_t>(blockIdx.x) * 2 * n;  // this CTA's level, trend
  float* vt = ell + n;
  auto step_scores = [&](int t) { return traj + (static_cast<size_t>(t) * rows + row) * stride; };

  // the first step initialises the state; every pass also ranks the next step's prediction
  KeyStats sp;
  {
    const float* IS = step_scores(0);
    for (int j = tid; j < n; j += kCalibThreads) {
      float l, v;
      ema_step(__ldg(IS + j), 0.f, 0.f, DSA_EMA_INIT, alpha, beta, l, v);
      ell[j] = l;
      vt[j] = v;
      keys[j] = score_key(ema_predict(l, v, gamma));
      sp.add(keys[j]);
    }
  }
  double total = 0.0;
  bool use_cand = false;  // the candidates of this step's P were collected by the last pass
  for (int t = 1; t < T; ++t) {
    const float* IS = step_scores(t);
    // P = the top-k_pred pages of the prediction made before step t's scores are seen: ranked
    // among the collected candidates when there are few enough, else from every key
    for (int w = tid; w < nwords; w += kCalibThreads) bitsP[w] = 0u;
    __syncthreads();
    int nP;
    if (use_cand) {
      nP = topk_candidates<kCalibThreads>(s_nc, k_pred, n, listP, ts);
    } else {
      nP = select_topk_block<kCalibThreads>(keys, n, k_pred, listP, sh, sp);
    }
    __syncthreads();
    for (int i = tid; i < nP; i += kCalibThreads) {
      const int j = listP[i];
      atomicOr(&bitsP[j >> 5], 1u << (j & 31));
    }
    __syncthreads();
    // the share of A_t's score mass that P covers (1 when A_t's scores sum to 0): one warp
    // (|A_t| <= 256, and double arithmetic is scarce)
    if (tid < 32) {
      const size_t ra = static_cast<size_t>(t) * rows + row;
      const int nA = min(max(__ldg(a_cnt + ra), 0), k);
      double num = 0.0, den = 0.0;
      for (int i = tid; i < nA; i += 32) {
        const int j = __ldg(a_idx + ra * k + i);
        const double s = __ldg(IS + j);
        den += s;
        if ((bitsP[j >> 5] >> (j & 31)) & 1u) num += s;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        num += __shfl_xor_sync(0xffffffffu, num, o);
        den += __shfl_xor_sync(0xffffffffu, den, o);
      }
      total += den != 0.0 ? num / den : 1.0;  // the same in every lane of warp 0
    }
    if (t == T - 1) break;
    // The predictor sees step t's scores and predicts step t + 1.  The k_pred pages of P_t keep
    // their new predictions at or above the smallest of them, so the next k_pred-th largest
    // prediction is at or above it too: the pages predicted at or above that bound are collected
    // while updating, and only they are ranked next step (when every page of P_t has a
    // prediction and at most kTopkMaxCand pages pass).
    if (tid == 0) {
      s_bound = 0xffffffffu;
      s_nc = 0;
    }
    __syncthreads();
    for (int i = tid; i < nP; i += kCalibThreads) {
      const int j = listP[i];
      float l, v;
      ema_step(__ldg(IS + j), ell[j], vt[j], DSA_EMA_UPDATE, alpha, beta, l, v);
      atomicMin(&s_bound, score_key(ema_predict(l, v, gamma)));
    }
    __syncthreads();
    const uint32_t bound = nP == k_pred ? s_bound : 0u;  // 0: no bound (a key of 0 is no page)
    sp = KeyStats();
    constexpr int kU = 4;  // items per thread whose loads are in flight together
    for (int j0 = 0; j0 < n; j0 += kU * kCalibThreads) {  // warp-uniform trip counts (ballots)
      float is[kU], lo[kU], vo[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u * kCalibThreads + tid;
        if (j < n) {
          is[u] = __ldg(IS + j);
          lo[u] = ell[j];
          vo[u] = vt[j];
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = j0 + u * kCalibThreads + tid;
        uint32_t key = 0u;
        if (j < n) {
          float l, v;
          ema_step(is[u], lo[u], vo[u], DSA_EMA_UPDATE, alpha, beta, l, v);
          ell[j] = l;
          vt[j] = v;
          key = score_key(ema_predict(l, v, gamma));
          keys[j] = key;
          sp.add(key);
        }
        const bool cand = bound != 0u && key >= bound && key != 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, cand);
        if (bal == 0u) continue;
        int at0 = 0;
        if (lane == 0) at0 = atomicAdd(&s_nc, __popc(bal));
        at0 = __shfl_sync(0xffffffffu, at0, 0);
        const int at = at0 + __popc(bal & ((1u << lane) - 1u));
        if (cand && at < kTopkMaxCand) {
          ts.ckey[at] = key;
          ts.cidx[at] = j;
        }
      }
    }
    __syncthreads();
    use_cand = bound != 0u && s_nc <= kTopkMaxCand;
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

size_t calib_smem_bytes(int n) { return static_cast<size_t>(n) * 4; }

CalibWorkspace calib_workspace(int T, int rows, int n, int k) {
  auto up16 = [](size_t x) { return (x + 15) & ~static_cast<size_t>(15); };
  CalibWorkspace w;
  w.done_off = 0;
  w.cnt_off = up16(static_cast<size_t>(rows) * 4);
  w.idx_off = w.cnt_off + up16(static_cast<size_t>(T) * rows * 4);
  w.state_off = w.idx_off + up16(static_cast<size_t>(T) * rows * k * 4);
  w.total = w.state_off + static_cast<size_t>(rows) * kCalibPoints * 2 * n * 4;
  return w;
}

cudaError_t launch_calib(const float* traj, int T, int rows, int n, int stride, int k, int k_pred,
                         float* H, int32_t* best, void* workspace, cudaStream_t s) {
  const CalibWorkspace w = calib_workspace(T, rows, n, k);
  char* ws = static_cast<char*>(workspace);
  int32_t* a_cnt = reinterpret_cast<int32_t*>(ws + w.cnt_off);
  int32_t* a_idx = reinterpret_cast<int32_t*>(ws + w.idx_off);
  // A_t of every (row, step): the trajectory is T * rows score rows of the same stride
  cudaError_t e = launch_select(traj, T * rows, n, stride, 1, k, a_idx, k, a_cnt, s);
  if (e != cudaSuccess) return e;
  const size_t bytes = calib_smem_bytes(n);
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(calib_kernel), bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(calib_kernel, rows * kCalibPoints, kCalibThreads, bytes, s, traj, T, rows, n,
                    stride, k, k_pred, a_idx, a_cnt, reinterpret_cast<float*>(ws + w.state_off), H,
                    best, reinterpret_cast<unsigned*>(ws + w.done_off));
}

}  // namespace dsa
