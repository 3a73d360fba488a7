// Internal launch interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <unordered_map>

#include "dsa.h"

namespace dsa {

constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 16;          // query heads per KV head served by one m16 tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxListPages = 256;     // pages one attention CTA may be handed
constexpr int kRecordFloats = 132;     // partial record: O[128], m, l, pad, pad
constexpr int kMaxSelectN = 32768;     // candidates per row held in shared memory by selection
constexpr int kMaxThresholdN = 16384;  // candidates per row for the PSA kernel

// Launches `kernel` as a programmatic dependent of the previous kernel in the stream: its blocks
// may be scheduled while that kernel finishes.  Every kernel of the library starts with
// launch_dependents() and grid_dependency_wait() (common.cuh), so it touches no global memory
// before the kernels ahead of it in the stream have completed.
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
}

struct KvView {
  const int32_t* page_table;
  const int32_t* seq_lens;
  const uint8_t* streaming;  // may be null
  int32_t* status;           // may be null
  int B, Hq, Hkv, G, D, p, max_pages, num_phys;
};

enum AttnList { LIST_SELECTED = 0, LIST_ONE_PAGE = 1, LIST_STREAMING = 2, LIST_REPAIR = 3 };

struct AttnArgs {
  KvView kv;
  const __nv_bfloat16* q;
  float scale_log2;
  const int32_t* idx;  // SELECTED / ONE_PAGE: selected positions; REPAIR: true set A
  int idx_stride;
  const int32_t* count;
  const int32_t* spec_idx;  // REPAIR: speculative set P
  int spec_stride;
  const int32_t* spec_count;
  int num_splits;
  int sink, local;  // STREAMING window
  float* out;
  float* m;
  float* l;
  float* part;  // partial records [rows][part_slots][G][kRecordFloats]
  int part_slots;
  int stages;
};

// Raises a kernel's dynamic shared-memory limit once per (kernel, device); later calls with the
// same or a smaller size do nothing, so steady-state launches (and stream capture) skip it.
inline cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, size_t> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) dev = 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done[dev].find(fn);
  if (it != done[dev].end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess) done[dev][fn] = bytes;
  return e;
}

size_t attn_smem_bytes(int page, int stages, int scratch_ints);
cudaError_t launch_attn(int list, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        const AttnArgs& a, int grid_x, cudaStream_t s);

struct MergeArgs {
  const float* part;  // [rows][slots][G][kRecordFloats]
  int slots;
  const int32_t* count;  // parts per row (null = slots)
  // repair: extra parts from page partials of hits
  const float* spec_part;
  int spec_stride;
  const int32_t* spec_idx;
  const int32_t* spec_count;
  const int32_t* true_idx;
  int true_stride;
  const int32_t* true_count;
  int superset;
  int rows, G, Hkv, Hq;
  const uint8_t* streaming;  // rows of streaming heads are skipped when non-null
  float* out;
  float* m;
  float* l;
  int out_rows_are_heads;  // 1: out index = (b*Hq + h*G + g); 0: out index = row*G + g
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s);

// Persistent split-K attention: CTAs take equal ranges of the global page-slot space; rows cut
// across CTAs are merged by the CTA that takes the row's last ticket.
struct StreamAttnArgs {
  KvView kv;
  const __nv_bfloat16* q;
  float scale_log2;
  const int32_t* idx;
  int idx_stride;
  const int32_t* count;
  int stages;
  float* part;        // [grid][2][G][kRecordFloats]: each CTA's first-row and last-row records
  int32_t* counters;  // [rows], zero on entry; left zero
  float* out;
  float* m;
  float* l;
  // streaming heads in the same launch: their sink + local tokens as extra units of
  // stream_stride slots each (0: streaming heads are skipped)
  int sink, local, stream_stride;
  // quantised pages instead of the bf16 pools (non-null): one block per (page, KV head) of
  // 264 p bytes (qbits 8, KV8) or 136 p bytes (qbits 4, KV4)
  const uint8_t* qkv;
  int qbits;
};
constexpr int kStreamMaxStages = 64;  // ring stages of the persistent attention (a 64-bit mask)
constexpr int kStreamMaxGrid = 512;  // bounds the row merge's [G][parts] weights in shared memory
size_t stream_attn_smem_bytes(int page, int stages, int G, int qbits = 0);  // qbits 0: bf16
int stream_attn_grid();  // CTAs of one launch: one per SM
cudaError_t launch_stream_attn(const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const StreamAttnArgs& a, int grid, cudaStream_t s);

// One PRR decode step in one launch of one CTA per SM (prr_step.cu).
constexpr int kPrrPredMax = 256;   // bound of k and k_pred
constexpr size_t kPrrSmemLimit = 227 * 1024;
struct PrrStepArgs {
  KvView kv;
  const __nv_bfloat16* kpool;
  const __nv_bfloat16* vpool;
  const __nv_bfloat16* q;
  const uint8_t* meta;  // MINMAX, logical page = page
  float* scores;
  int stride;
  float* ell;
  float* trend;
  float alpha, beta, gamma;
  float* pred;
  const int32_t* spec_idx;
  const int32_t* spec_count;
  int k_pred;
  float* partials;
  int32_t* idx;
  int32_t* count;
  int k;
  int32_t* next_idx;
  int32_t* next_count;
  int superset;
  float scale_log2;
  float* out;
  float* m;
  float* l;
};
// shared memory of one launch (SIZE_MAX when no ring depth fits)
size_t prr_step_smem_bytes(int page, int n, int k_pred);
// workspace: per-row counters first (prr_step_counter_bytes of them, zero on entry, left zero),
// then the new predictions [rows][max_pages]
size_t prr_step_workspace_bytes(int rows, int max_pages);
size_t prr_step_counter_bytes(int rows);
cudaError_t launch_prr_step(const CUtensorMap& tmK, const CUtensorMap& tmV, const PrrStepArgs& a,
                            void* workspace, cudaStream_t s);

// metadata and scoring
cudaError_t launch_build_meta(const KvView& kv, const __nv_bfloat16* k_pages, int kind, int lp,
                              void* meta, cudaStream_t s);
cudaError_t launch_append_kv(const KvView& kv, __nv_bfloat16* k_pages, __nv_bfloat16* v_pages,
                             const __nv_bfloat16* k_new, const __nv_bfloat16* v_new, int kind,
                             int lp, void* meta, cudaStream_t s);
cudaError_t launch_score(const KvView& kv, const __nv_bfloat16* q, const void* meta, int kind,
                         int lp, float* scores, int stride, cudaStream_t s);

// selection
cudaError_t launch_select(const float* scores, int rows, int n_logical, int stride, int g, int k,
                          int32_t* idx, int idx_stride, int32_t* count, cudaStream_t s);
cudaError_t launch_ema(const float* IS, int rows, int n, int stride, float* ell, float* v,
                       int mode, float alpha, float beta, float gamma, float* pred, int k_pred,
                       int32_t* pred_idx, int pred_idx_stride, int32_t* pred_count,
                       cudaStream_t s);

// Quantised KV pages (kvquant.cu): KV8 (e4m3) or KV4 (4-bit integer) codes of K and V with an
// fp32 scale per (page, KV head, token) row
cudaError_t launch_quantize_kv8(const __nv_bfloat16* src, long long n_rows, int page, int v,
                                uint8_t* kv8, cudaStream_t s);
cudaError_t launch_quantize_kv4(const __nv_bfloat16* src, long long n_rows, int page, int v,
                                uint8_t* kv4, cudaStream_t s);

// PRR §3.2 calibration of the EMA predictor over its 80-point grid (csrc/calib.cu)
constexpr int kCalibPoints = 80;
constexpr int kCalibMaxN = 16384;  // pages per row whose predictor state fits in shared memory
size_t calib_smem_bytes(int n);
// workspace: per-row counters, A_t of every (step, row) (counts, indices), the predictor state of
// every (row, grid point)
struct CalibWorkspace {
  size_t done_off, cnt_off, idx_off, state_off, total;
};
CalibWorkspace calib_workspace(int T, int rows, int n, int k);
cudaError_t launch_calib(const float* traj, int T, int rows, int n, int stride, int k, int k_pred,
                         float* H, int32_t* best, void* workspace, cudaStream_t s);

struct ThresholdArgs {
  KvView kv;
  const __nv_bfloat16* q;
  const float* scores;
  int score_stride;
  float tau;
  int cap;
  int flags;
  float scale_log2;
  int32_t* idx;
  int idx_stride;
  int32_t* count;
  float* out;
  float* m;
  float* l;
};
cudaError_t launch_threshold(const CUtensorMap& tmK, const CUtensorMap& tmV,
                             const ThresholdArgs& a, cudaStream_t s);

}  // namespace dsa
