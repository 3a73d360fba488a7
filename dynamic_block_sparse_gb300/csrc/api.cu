// C ABI of libdsa: validates arguments on the host, encodes TMA descriptors for the KV pools,
// chooses split counts and launches the kernels on the caller's stream.  Allocates nothing.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "internal.h"

namespace dsa {
size_t threshold_smem_bytes(int page, int max_pages);
}

namespace {

using namespace dsa;

constexpr int kTargetCtas = 2 * 152;  // two CTAs per SM of a GB300

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int ok() {
  g_err.clear();
  return DSA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D view of a pool: (64 dims, token rows, 2 halves) with strides 256 B per token row and 128 B
// per half, so one box of (64, page, 2) with 128-byte swizzle stages a whole page of one KV head:
// dims 0..63 of its rows, then dims 64..127 of its rows.
int pool_map(const void* base, const dsa_paged_kv* kv, CUtensorMap* map) {
  auto fn = encode_fn();
  if (!fn) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {64,
                        static_cast<cuuint64_t>(kv->num_phys_pages) * kv->num_kv_heads *
                            kv->page_size,
                        2};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kv->page_size), 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return DSA_OK;
}

// Checks the cache descriptor.  pools: whether k/v pools are needed (0 none, 1 K only, 2 both).
int check_kv(const dsa_paged_kv* kv, int pools, KvView* view) {
  if (!kv) return fail(DSA_ERR_INVALID_ARG, "kv descriptor is NULL");
  if (!kv->page_table || !kv->seq_lens) return fail(DSA_ERR_INVALID_ARG, "page_table/seq_lens NULL");
  if (pools >= 1 && !kv->k_pages) return fail(DSA_ERR_INVALID_ARG, "k_pages is NULL");
  if (pools >= 2 && !kv->v_pages) return fail(DSA_ERR_INVALID_ARG, "v_pages is NULL");
  if (kv->batch <= 0 || kv->num_q_heads <= 0 || kv->num_kv_heads <= 0 || kv->page_size <= 0 ||
      kv->max_pages_per_seq <= 0 || kv->num_phys_pages <= 0)
    return fail(DSA_ERR_INVALID_ARG, "kv shape fields must be positive");
  if (kv->head_dim != kHeadDim)
    return fail(DSA_ERR_UNSUPPORTED, "head_dim %d unsupported (only 128)", kv->head_dim);
  if (kv->num_q_heads % kv->num_kv_heads != 0)
    return fail(DSA_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
  const int G = kv->num_q_heads / kv->num_kv_heads;
  if (G > kMaxGroup) return fail(DSA_ERR_UNSUPPORTED, "group size %d > %d", G, kMaxGroup);
  if (kv->page_size % 16 != 0 || kv->page_size > 256)
    return fail(DSA_ERR_UNSUPPORTED, "page_size %d must be a multiple of 16 in [16, 256]",
                kv->page_size);
  const long long rows =
      static_cast<long long>(kv->num_phys_pages) * kv->num_kv_heads * kv->page_size;
  if (rows >= (1LL << 31))
    return fail(DSA_ERR_UNSUPPORTED, "pool of %lld token rows exceeds 2^31", rows);
  if ((pools >= 1 && !aligned(kv->k_pages, 16)) || (pools >= 2 && !aligned(kv->v_pages, 16)))
    return fail(DSA_ERR_ALIGNMENT, "k_pages/v_pages must be 16-byte aligned");
  view->page_table = kv->page_table;
  view->seq_lens = kv->seq_lens;
  view->streaming = kv->head_is_streaming;
  view->status = kv->status;
  view->B = kv->batch;
  view->Hq = kv->num_q_heads;
  view->Hkv = kv->num_kv_heads;
  view->G = G;
  view->D = kv->head_dim;
  view->p = kv->page_size;
  view->max_pages = kv->max_pages_per_seq;
  view->num_phys = kv->num_phys_pages;
  return DSA_OK;
}

int attn_stages(int page, int pages_per_cta) {
  int s = 131072 / (512 * page);
  if (s < 1) s = 1;
  if (s > 8) s = 8;
  if (pages_per_cta >= 1 && s > pages_per_cta) s = pages_per_cta;
  return s;
}

int auto_splits(int rows, int stride, int requested) {
  int min_splits = (stride + kMaxListPages - 1) / kMaxListPages;
  if (min_splits < 1) min_splits = 1;
  int s = requested;
  if (s <= 0) {
    s = (kTargetCtas + rows - 1) / rows;
    const int cap = (stride + 1) / 2;  // at least two pages per CTA on average
    if (s > cap) s = cap;
  }
  if (s < min_splits) s = min_splits;
  if (s > stride && stride > 0) s = stride;
  if (s < 1) s = 1;
  return s;
}

int repair_splits(int stride) {
  int s = (stride + 3) / 4;
  const int min_splits = (stride + kMaxListPages - 1) / kMaxListPages;
  if (s < min_splits) s = min_splits;
  return s < 1 ? 1 : s;
}

// Workspace of the persistent split-K path: two partial records per CTA of its grid, then one
// ticket counter per row.
size_t stream_records_bytes(int grid, int G) {
  const size_t rec = static_cast<size_t>(grid) * 2 * G * kRecordFloats * sizeof(float);
  return (rec + 255) & ~static_cast<size_t>(255);
}

size_t stream_workspace_bytes(int rows, int grid, int G) {
  return stream_records_bytes(grid, G) + static_cast<size_t>(rows) * sizeof(int32_t);
}

size_t record_bytes(int rows, int slots, int G) {
  return static_cast<size_t>(rows) * slots * G * kRecordFloats * sizeof(float);
}

float scale_log2(float scale) { return scale * kLog2e; }

}  // namespace

// ---------------------------------------------------------------------------------------------
// Fixed scratch for dsa_sparse_decode_attn_noalloc.  Some callers cannot call cudaMalloc: code
// that runs inside a host framework which owns all device memory through its own allocator, and
// latency-critical loops where the implicit device synchronisation of cudaMalloc/cudaFree is not
// acceptable.  For them the split-K partial records live in this array, which every GPU that
// loads the library holds until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_noalloc_scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device (with that device
// current) and cached.
int noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    addr[dev] = p;
  }
  *out = addr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" {

const char* dsa_last_error(void) { return g_err.c_str(); }

const char* dsa_version(void) { return "libdsa 0.1 (sm_103a)"; }

int dsa_build_page_meta(const dsa_paged_kv* kv, int32_t meta_kind, int32_t logical_page,
                        void* meta, dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 1, &v);
  if (rc) return rc;
  if (meta_kind != DSA_META_MINMAX && meta_kind != DSA_META_MEAN)
    return fail(DSA_ERR_INVALID_ARG, "unknown meta_kind %d", meta_kind);
  if (logical_page <= 0 || v.p % logical_page != 0)
    return fail(DSA_ERR_INVALID_ARG, "logical_page %d must divide page_size %d", logical_page, v.p);
  if (!meta) return fail(DSA_ERR_INVALID_ARG, "meta is NULL");
  if (!aligned(meta, 16)) return fail(DSA_ERR_ALIGNMENT, "meta must be 16-byte aligned");
  cudaError_t e = launch_build_meta(v, static_cast<const __nv_bfloat16*>(kv->k_pages), meta_kind,
                                    logical_page, meta, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_build_page_meta launch");
}

int dsa_append_kv(const dsa_paged_kv* kv, const void* k_new, const void* v_new,
                  int32_t meta_kind, int32_t logical_page, void* meta, dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 1, &v);
  if (rc) return rc;
  if (!k_new || !v_new) return fail(DSA_ERR_INVALID_ARG, "k_new/v_new is NULL");
  if (!aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(DSA_ERR_ALIGNMENT, "k_new/v_new must be 16-byte aligned");
  if (meta) {
    if (meta_kind != DSA_META_MINMAX && meta_kind != DSA_META_MEAN)
      return fail(DSA_ERR_INVALID_ARG, "unknown meta_kind %d", meta_kind);
    if (logical_page <= 0 || v.p % logical_page != 0)
      return fail(DSA_ERR_INVALID_ARG, "logical_page %d must divide page_size %d", logical_page,
                  v.p);
    if (!aligned(meta, 16)) return fail(DSA_ERR_ALIGNMENT, "meta must be 16-byte aligned");
  }
  // the pools are the caller's, written here (the struct's pointers are const for the readers)
  cudaError_t e = launch_append_kv(
      v, static_cast<__nv_bfloat16*>(const_cast<void*>(kv->k_pages)),
      static_cast<__nv_bfloat16*>(const_cast<void*>(kv->v_pages)),
      static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
      meta_kind, logical_page, meta, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_append_kv launch");
}

int dsa_score_pages(const dsa_paged_kv* kv, const void* q, const void* meta, int32_t meta_kind,
                    int32_t logical_page, float* scores, int32_t score_stride,
                    dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 0, &v);
  if (rc) return rc;
  if (!q || !meta || !scores) return fail(DSA_ERR_INVALID_ARG, "q/meta/scores is NULL");
  if (meta_kind != DSA_META_MINMAX && meta_kind != DSA_META_MEAN)
    return fail(DSA_ERR_INVALID_ARG, "unknown meta_kind %d", meta_kind);
  if (logical_page <= 0 || v.p % logical_page != 0)
    return fail(DSA_ERR_INVALID_ARG, "logical_page %d must divide page_size %d", logical_page, v.p);
  if (!aligned(meta, 16)) return fail(DSA_ERR_ALIGNMENT, "meta must be 16-byte aligned");
  const long long need = static_cast<long long>(v.max_pages) * (v.p / logical_page);
  if (score_stride < need)
    return fail(DSA_ERR_INVALID_ARG, "score_stride %d < max_pages * g = %lld", score_stride, need);
  cudaError_t e = launch_score(v, static_cast<const __nv_bfloat16*>(q), meta, meta_kind,
                               logical_page, scores, score_stride,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_score_pages launch");
}

static int select_common(const float* scores, int32_t rows, int32_t n_logical, int32_t stride,
                         int32_t g, int32_t k, int32_t* idx, int32_t idx_stride, int32_t* count,
                         dsa_stream_t stream, const char* name) {
  if (rows < 0 || n_logical < 0 || k < 0 || g < 1)
    return fail(DSA_ERR_INVALID_ARG, "%s: negative size or g < 1", name);
  if (rows == 0) return ok();
  if (!scores || !idx || !count) return fail(DSA_ERR_INVALID_ARG, "%s: NULL pointer", name);
  if (n_logical > stride) return fail(DSA_ERR_INVALID_ARG, "%s: n > stride", name);
  if (idx_stride < k) return fail(DSA_ERR_INVALID_ARG, "%s: idx_stride < k", name);
  const int n = (n_logical + g - 1) / g;
  if (n > kMaxSelectN)
    return fail(DSA_ERR_UNSUPPORTED, "%s: %d candidates per row > %d", name, n, kMaxSelectN);
  cudaError_t e = launch_select(scores, rows, n_logical, stride, g, k, idx, idx_stride, count,
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, name);
}

int dsa_select_topk(const float* scores, int32_t rows, int32_t n, int32_t stride, int32_t k,
                    int32_t* idx, int32_t idx_stride, int32_t* count, dsa_stream_t stream) {
  return select_common(scores, rows, n, stride, 1, k, idx, idx_stride, count, stream,
                       "dsa_select_topk");
}

int dsa_select_hier(const float* logical_scores, int32_t rows, int32_t n_logical, int32_t stride,
                    int32_t g, int32_t k_phys, int32_t* idx, int32_t idx_stride, int32_t* count,
                    dsa_stream_t stream) {
  return select_common(logical_scores, rows, n_logical, stride, g, k_phys, idx, idx_stride, count,
                       stream, "dsa_select_hier");
}

int dsa_select_threshold(const dsa_paged_kv* kv, const void* q, const float* scores,
                         int32_t score_stride, float tau, int32_t cap, int32_t flags, float scale,
                         int32_t* idx, int32_t idx_stride, int32_t* count, float* out, float* m,
                         float* l, dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!q || !scores || !idx || !count || !out || !m || !l)
    return fail(DSA_ERR_INVALID_ARG, "dsa_select_threshold: NULL pointer");
  if (!(tau > 0.f && tau <= 1.f)) return fail(DSA_ERR_INVALID_ARG, "tau must be in (0, 1]");
  if (!aligned(q, 16)) return fail(DSA_ERR_ALIGNMENT, "q must be 16-byte aligned");
  if (cap < 1 || idx_stride < cap) return fail(DSA_ERR_INVALID_ARG, "need 1 <= cap <= idx_stride");
  if (score_stride < 1) return fail(DSA_ERR_INVALID_ARG, "score_stride < 1");
  if (v.max_pages > kMaxThresholdN)
    return fail(DSA_ERR_UNSUPPORTED, "max_pages_per_seq %d > %d for threshold selection",
                v.max_pages, kMaxThresholdN);
  if (threshold_smem_bytes(v.p, v.max_pages) > 227 * 1024)
    return fail(DSA_ERR_UNSUPPORTED, "threshold selection shared memory too large");
  CUtensorMap tk, tv;
  if ((rc = pool_map(kv->k_pages, kv, &tk)) || (rc = pool_map(kv->v_pages, kv, &tv))) return rc;
  ThresholdArgs a;
  a.kv = v;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scores = scores;
  a.score_stride = score_stride;
  a.tau = tau;
  a.cap = cap;
  a.flags = flags;
  a.scale_log2 = scale_log2(scale);
  a.idx = idx;
  a.idx_stride = idx_stride;
  a.count = count;
  a.out = out;
  a.m = m;
  a.l = l;
  cudaError_t e = launch_threshold(tk, tv, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_select_threshold launch");
}

size_t dsa_sparse_decode_attn_workspace_size(const dsa_paged_kv* kv, int32_t idx_stride,
                                             int32_t num_splits) {
  if (!kv || kv->num_kv_heads <= 0 || kv->batch <= 0 || idx_stride <= 0) return 0;
  const int rows = kv->batch * kv->num_kv_heads;
  const int G = kv->num_q_heads / kv->num_kv_heads;
  const int s = auto_splits(rows, idx_stride, num_splits);
  const size_t classic = s > 1 ? record_bytes(rows, s, G) : 0;
  if (num_splits > 0) return classic;
  const size_t streamed = stream_workspace_bytes(rows, stream_attn_grid(), G);
  return classic > streamed ? classic : streamed;
}

int dsa_hybrid_decode_attn(const dsa_paged_kv* kv, const void* q, const int32_t* idx,
                           int32_t idx_stride, const int32_t* count, int32_t sink_tokens,
                           int32_t local_tokens, float scale, float* out, float* m, float* l,
                           void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!q || !idx || !count || !out || !m || !l)
    return fail(DSA_ERR_INVALID_ARG, "q/idx/count/out/m/l is NULL");
  if (idx_stride < 1) return fail(DSA_ERR_INVALID_ARG, "idx_stride < 1");
  if (sink_tokens < 0 || local_tokens < 0)
    return fail(DSA_ERR_INVALID_ARG, "negative sink/local tokens");
  if (!aligned(q, 16) || !aligned(out, 16))
    return fail(DSA_ERR_ALIGNMENT, "q and out must be 16-byte aligned");
  if (v.Hkv > 1024) return fail(DSA_ERR_UNSUPPORTED, "more than 1024 KV heads");
  // pages a streaming row may touch: those of its sink tokens and of its local window
  const long long sslots = (static_cast<long long>(sink_tokens) + v.p - 1) / v.p +
                           (static_cast<long long>(local_tokens) + v.p - 1) / v.p + 1;
  if (sslots > 65536) return fail(DSA_ERR_UNSUPPORTED, "sink/local window too long");
  const int grid = stream_attn_grid();
  const int rows = v.B * v.Hkv;
  const size_t rec = stream_records_bytes(grid, v.G);
  const size_t need = stream_workspace_bytes(rows, grid, v.G);
  if (!workspace || workspace_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return fail(DSA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  CUtensorMap tk, tv;
  if ((rc = pool_map(kv->k_pages, kv, &tk)) || (rc = pool_map(kv->v_pages, kv, &tv))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int stages = 131072 / (512 * v.p);
  if (stages < 1) stages = 1;
  if (stages > kStreamMaxStages) stages = kStreamMaxStages;
  StreamAttnArgs sa = {};
  sa.kv = v;
  sa.q = static_cast<const __nv_bfloat16*>(q);
  sa.scale_log2 = scale_log2(scale);
  sa.idx = idx;
  sa.idx_stride = idx_stride;
  sa.count = count;
  sa.stages = stages;
  sa.part = static_cast<float*>(workspace);
  sa.counters = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + rec);
  sa.out = out;
  sa.m = m;
  sa.l = l;
  sa.sink = sink_tokens;
  sa.local = local_tokens;
  sa.stream_stride = v.streaming != nullptr ? static_cast<int>(sslots) : 0;
  // the row tickets are zero on entry (zero-filled workspace, left zero by every completed call)
  const cudaError_t e = launch_stream_attn(tk, tv, sa, grid, s);
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_hybrid_decode_attn launch");
}

int dsa_sparse_decode_attn(const dsa_paged_kv* kv, const void* q, const int32_t* idx,
                           int32_t idx_stride, const int32_t* count, float scale, float* out,
                           float* m, float* l, float* page_partials, int32_t num_splits,
                           void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!q || !idx || !count) return fail(DSA_ERR_INVALID_ARG, "q/idx/count is NULL");
  if (idx_stride < 1) return fail(DSA_ERR_INVALID_ARG, "idx_stride < 1");
  if (!aligned(q, 16)) return fail(DSA_ERR_ALIGNMENT, "q must be 16-byte aligned");
  if (page_partials && !aligned(page_partials, 16))
    return fail(DSA_ERR_ALIGNMENT, "page_partials must be 16-byte aligned");
  const bool want_out = out != nullptr;
  if (want_out && (!m || !l)) return fail(DSA_ERR_INVALID_ARG, "out given without m/l");
  if (!want_out && !page_partials)
    return fail(DSA_ERR_INVALID_ARG, "neither out nor page_partials given");
  CUtensorMap tk, tv;
  if ((rc = pool_map(kv->k_pages, kv, &tk)) || (rc = pool_map(kv->v_pages, kv, &tv))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rows = v.B * v.Hkv;
  AttnArgs a = {};
  a.kv = v;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scale_log2 = scale_log2(scale);
  a.idx = idx;
  a.idx_stride = idx_stride;
  a.count = count;
  cudaError_t e;
  if (page_partials) {
    a.num_splits = idx_stride;
    a.part = page_partials;
    a.part_slots = idx_stride;
    a.stages = 1;
    e = launch_attn(LIST_ONE_PAGE, tk, tv, a, idx_stride, s);
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_decode_attn launch");
    if (want_out) {
      MergeArgs mg = {};
      mg.part = page_partials;
      mg.slots = idx_stride;
      mg.count = count;
      mg.rows = rows;
      mg.G = v.G;
      mg.Hkv = v.Hkv;
      mg.Hq = v.Hq;
      mg.streaming = v.streaming;
      mg.out = out;
      mg.m = m;
      mg.l = l;
      mg.out_rows_are_heads = 1;
      e = launch_merge(mg, s);
      if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_decode_attn merge");
    }
    return ok();
  }
  // default: one persistent launch; the last unit of each row merges it
  if (num_splits <= 0 && want_out && v.Hkv <= 1024) {
    if (!aligned(out, 16)) return fail(DSA_ERR_ALIGNMENT, "out must be 16-byte aligned");
    const int grid = stream_attn_grid();
    const size_t rec = stream_records_bytes(grid, v.G);
    const size_t need = stream_workspace_bytes(rows, grid, v.G);
    if (!workspace || workspace_bytes < need)
      return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
    if (!aligned(workspace, 16)) return fail(DSA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
    int stages = 131072 / (512 * v.p);
    if (stages < 1) stages = 1;
    if (stages > kStreamMaxStages) stages = kStreamMaxStages;
    StreamAttnArgs sa = {};
    sa.kv = v;
    sa.q = a.q;
    sa.scale_log2 = a.scale_log2;
    sa.idx = idx;
    sa.idx_stride = idx_stride;
    sa.count = count;
    sa.stages = stages;
    sa.part = static_cast<float*>(workspace);
    sa.counters = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + rec);
    sa.out = out;
    sa.m = m;
    sa.l = l;
    // the row tickets are zero on entry (zero-filled workspace, left zero by every completed call)
    e = launch_stream_attn(tk, tv, sa, grid, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_sparse_decode_attn launch");
  }
  const int splits = auto_splits(rows, idx_stride, num_splits);
  const int per_cta = (idx_stride + splits - 1) / splits;
  a.num_splits = splits;
  a.stages = attn_stages(v.p, per_cta);
  a.out = out;
  a.m = m;
  a.l = l;
  if (splits > 1) {
    const size_t need = record_bytes(rows, splits, v.G);
    if (!workspace || workspace_bytes < need)
      return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
    if (!aligned(workspace, 16)) return fail(DSA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
    a.part = static_cast<float*>(workspace);
    a.part_slots = splits;
  }
  e = launch_attn(LIST_SELECTED, tk, tv, a, splits, s);
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_decode_attn launch");
  if (splits > 1) {
    MergeArgs mg = {};
    mg.part = static_cast<const float*>(workspace);
    mg.slots = splits;
    mg.rows = rows;
    mg.G = v.G;
    mg.Hkv = v.Hkv;
    mg.Hq = v.Hq;
    mg.streaming = v.streaming;
    mg.out = out;
    mg.m = m;
    mg.l = l;
    mg.out_rows_are_heads = 1;
    e = launch_merge(mg, s);
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_decode_attn merge");
  }
  return ok();
}

size_t dsa_repair_merge_workspace_size(const dsa_paged_kv* kv, int32_t true_stride) {
  if (!kv || kv->num_kv_heads <= 0 || kv->batch <= 0 || true_stride <= 0) return 0;
  const int rows = kv->batch * kv->num_kv_heads;
  const int G = kv->num_q_heads / kv->num_kv_heads;
  return record_bytes(rows, repair_splits(true_stride), G);
}

int dsa_repair_merge(const dsa_paged_kv* kv, const void* q, const int32_t* spec_idx,
                     int32_t spec_stride, const int32_t* spec_count, const float* page_partials,
                     const int32_t* true_idx, int32_t true_stride, const int32_t* true_count,
                     int32_t superset, float scale, float* out, float* m, float* l,
                     void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!q || !spec_idx || !spec_count || !page_partials || !true_idx || !true_count || !out || !m ||
      !l)
    return fail(DSA_ERR_INVALID_ARG, "dsa_repair_merge: NULL pointer");
  if (spec_stride < 1 || true_stride < 1) return fail(DSA_ERR_INVALID_ARG, "stride < 1");
  if (!aligned(q, 16) || !aligned(page_partials, 16))
    return fail(DSA_ERR_ALIGNMENT, "q and page_partials must be 16-byte aligned");
  if (spec_stride > 8192 || true_stride > 8192)
    return fail(DSA_ERR_UNSUPPORTED, "repair lists longer than 8192 pages");
  const int rows = v.B * v.Hkv;
  const int splits = repair_splits(true_stride);
  const size_t need = record_bytes(rows, splits, v.G);
  if (!workspace || workspace_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return fail(DSA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  CUtensorMap tk, tv;
  if ((rc = pool_map(kv->k_pages, kv, &tk)) || (rc = pool_map(kv->v_pages, kv, &tv))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AttnArgs a = {};
  a.kv = v;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scale_log2 = scale_log2(scale);
  a.idx = true_idx;
  a.idx_stride = true_stride;
  a.count = true_count;
  a.spec_idx = spec_idx;
  a.spec_stride = spec_stride;
  a.spec_count = spec_count;
  a.num_splits = splits;
  a.part = static_cast<float*>(workspace);
  a.part_slots = splits;
  a.stages = attn_stages(v.p, (true_stride + splits - 1) / splits);
  cudaError_t e = launch_attn(LIST_REPAIR, tk, tv, a, splits, s);
  if (e != cudaSuccess) return cuda_fail(e, "dsa_repair_merge launch");
  MergeArgs mg = {};
  mg.part = static_cast<const float*>(workspace);
  mg.slots = splits;
  mg.spec_part = page_partials;
  mg.spec_stride = spec_stride;
  mg.spec_idx = spec_idx;
  mg.spec_count = spec_count;
  mg.true_idx = true_idx;
  mg.true_stride = true_stride;
  mg.true_count = true_count;
  mg.superset = superset != 0;
  mg.rows = rows;
  mg.G = v.G;
  mg.Hkv = v.Hkv;
  mg.Hq = v.Hq;
  mg.streaming = v.streaming;
  mg.out = out;
  mg.m = m;
  mg.l = l;
  mg.out_rows_are_heads = 1;
  e = launch_merge(mg, s);
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_repair_merge merge");
}

int dsa_streaming_head_attn(const dsa_paged_kv* kv, const void* q, int32_t sink_tokens,
                            int32_t local_tokens, float scale, float* out, float* m, float* l,
                            dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!q || !out || !m || !l) return fail(DSA_ERR_INVALID_ARG, "q/out/m/l is NULL");
  if (sink_tokens < 0 || local_tokens < 0) return fail(DSA_ERR_INVALID_ARG, "negative window");
  if (!aligned(q, 16)) return fail(DSA_ERR_ALIGNMENT, "q must be 16-byte aligned");
  if (!kv->head_is_streaming) return ok();  // no streaming heads: nothing to do
  const long long pages = (static_cast<long long>(sink_tokens) + v.p - 1) / v.p +
                          (static_cast<long long>(local_tokens) + v.p - 1) / v.p + 1;
  if (pages > kMaxListPages)
    return fail(DSA_ERR_UNSUPPORTED, "sink + local spans more than %d pages", kMaxListPages);
  CUtensorMap tk, tv;
  if ((rc = pool_map(kv->k_pages, kv, &tk)) || (rc = pool_map(kv->v_pages, kv, &tv))) return rc;
  AttnArgs a = {};
  a.kv = v;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scale_log2 = scale_log2(scale);
  a.num_splits = 1;
  a.sink = sink_tokens;
  a.local = local_tokens;
  a.out = out;
  a.m = m;
  a.l = l;
  a.stages = attn_stages(v.p, static_cast<int>(pages));
  cudaError_t e = launch_attn(LIST_STREAMING, tk, tv, a, 1, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_streaming_head_attn launch");
}

int dsa_ema_predict_update(const float* IS, int32_t rows, int32_t n, int32_t stride, float* ell,
                           float* v, int32_t mode, float alpha, float beta, float gamma,
                           float* pred, int32_t k_pred, int32_t* pred_idx,
                           int32_t pred_idx_stride, int32_t* pred_count, dsa_stream_t stream) {
  if (rows < 0 || n < 0 || k_pred < 0) return fail(DSA_ERR_INVALID_ARG, "negative size");
  if (rows == 0) return ok();
  if (!IS || !ell || !v) return fail(DSA_ERR_INVALID_ARG, "IS/ell/v is NULL");
  if (mode != DSA_EMA_INIT && mode != DSA_EMA_UPDATE)
    return fail(DSA_ERR_INVALID_ARG, "unknown EMA mode %d", mode);
  if (n > stride) return fail(DSA_ERR_INVALID_ARG, "n > stride");
  if (n > kMaxSelectN) return fail(DSA_ERR_UNSUPPORTED, "n %d > %d", n, kMaxSelectN);
  if (k_pred > 0 && (!pred_idx || !pred_count || pred_idx_stride < k_pred))
    return fail(DSA_ERR_INVALID_ARG, "pred_idx/pred_count NULL or pred_idx_stride < k_pred");
  cudaError_t e = launch_ema(IS, rows, n, stride, ell, v, mode, alpha, beta, gamma, pred, k_pred,
                             pred_idx, pred_idx_stride, pred_count,
                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_ema_predict_update launch");
}

}  // extern "C"

namespace {

// Both quantisers: every K row, then every V row of the pool into its block.
int quantize_pool(const dsa_paged_kv* kv, void* dst, int qbits, dsa_stream_t stream,
                  const char* name) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!dst) return fail(DSA_ERR_INVALID_ARG, "%s: the block buffer is NULL", name);
  if (!aligned(dst, 16)) return fail(DSA_ERR_ALIGNMENT, "%s: blocks must be 16-byte aligned", name);
  const long long n_rows = static_cast<long long>(v.num_phys) * v.Hkv * v.p;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto launch = qbits == 8 ? launch_quantize_kv8 : launch_quantize_kv4;
  cudaError_t e = launch(static_cast<const __nv_bfloat16*>(kv->k_pages), n_rows, v.p, 0,
                         static_cast<uint8_t*>(dst), s);
  if (e == cudaSuccess)
    e = launch(static_cast<const __nv_bfloat16*>(kv->v_pages), n_rows, v.p, 1,
               static_cast<uint8_t*>(dst), s);
  return e == cudaSuccess ? ok() : cuda_fail(e, name);
}

size_t pool_block_bytes(const dsa_paged_kv* kv, int per_token) {
  if (!kv || kv->num_phys_pages <= 0 || kv->num_kv_heads <= 0 || kv->page_size <= 0) return 0;
  return static_cast<size_t>(kv->num_phys_pages) * kv->num_kv_heads * kv->page_size * per_token;
}

// The persistent attention over quantised blocks (KV8 or KV4).
int quantized_attn(const dsa_paged_kv* kv, const void* blocks, int qbits, const void* q,
                   const int32_t* idx, int32_t idx_stride, const int32_t* count, float scale,
                   float* out, float* m, float* l, void* workspace, size_t workspace_bytes,
                   dsa_stream_t stream, const char* name) {
  KvView v;
  int rc = check_kv(kv, 0, &v);
  if (rc) return rc;
  if (!blocks || !q || !idx || !count || !out || !m || !l)
    return fail(DSA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
  if (idx_stride < 1) return fail(DSA_ERR_INVALID_ARG, "idx_stride < 1");
  if (!aligned(blocks, 16) || !aligned(q, 16) || !aligned(out, 16))
    return fail(DSA_ERR_ALIGNMENT, "%s: blocks, q and out must be 16-byte aligned", name);
  if (v.Hkv > 1024) return fail(DSA_ERR_UNSUPPORTED, "more than 1024 KV heads");
  const int rows = v.B * v.Hkv;
  const int grid = stream_attn_grid();
  const size_t rec = stream_records_bytes(grid, v.G);
  const size_t need = stream_workspace_bytes(rows, grid, v.G);
  if (!workspace || workspace_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return fail(DSA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  // as many stages (one page block each) as fit in 160 KB: the small blocks need many in flight
  // to keep the page rate of the bytes' roofline (stages / load latency)
  const size_t smem_cap = 227 * 1024;
  const int per_token = qbits == 8 ? 264 : 136;
  const int stride = (per_token * v.p + 15) & ~15;
  int stages = 163840 / stride;
  if (stages > kStreamMaxStages) stages = kStreamMaxStages;
  while (stages > 1 && stream_attn_smem_bytes(v.p, stages, v.G, qbits) > smem_cap) --stages;
  if (stages < 1 || stream_attn_smem_bytes(v.p, stages, v.G, qbits) > smem_cap)
    return fail(DSA_ERR_UNSUPPORTED, "%s: shape needs too much shared memory", name);
  // every consumer warp owns the same number of (stage, 16-token tile) slots of the ring
  const int tiles = v.p / 16;
  while (stages * tiles > 8 && (stages * tiles) % 8 != 0) --stages;
  StreamAttnArgs sa = {};
  sa.kv = v;
  sa.q = static_cast<const __nv_bfloat16*>(q);
  sa.scale_log2 = scale_log2(scale);
  sa.idx = idx;
  sa.idx_stride = idx_stride;
  sa.count = count;
  sa.stages = stages;
  sa.part = static_cast<float*>(workspace);
  sa.counters = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + rec);
  sa.out = out;
  sa.m = m;
  sa.l = l;
  sa.qkv = static_cast<const uint8_t*>(blocks);
  sa.qbits = qbits;
  // the row tickets are zero on entry (zero-filled workspace, left zero by every completed call)
  CUtensorMap none = {};  // quantised pages move by plain bulk copies: no tensor maps
  const cudaError_t e = launch_stream_attn(none, none, sa, grid, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, name);
}

size_t quantized_attn_workspace(const dsa_paged_kv* kv, int32_t idx_stride) {
  if (!kv || kv->num_kv_heads <= 0 || kv->batch <= 0 || idx_stride <= 0) return 0;
  const int rows = kv->batch * kv->num_kv_heads;
  const int G = kv->num_q_heads / kv->num_kv_heads;
  return stream_workspace_bytes(rows, stream_attn_grid(), G);
}

}  // namespace

extern "C" {

int dsa_quantize_kv8(const dsa_paged_kv* kv, void* kv8, dsa_stream_t stream) {
  return quantize_pool(kv, kv8, 8, stream, "dsa_quantize_kv8");
}

size_t dsa_kv8_bytes(const dsa_paged_kv* kv) { return pool_block_bytes(kv, 264); }

size_t dsa_sparse_decode_attn_kv8_workspace_size(const dsa_paged_kv* kv, int32_t idx_stride) {
  return quantized_attn_workspace(kv, idx_stride);
}

int dsa_sparse_decode_attn_kv8(const dsa_paged_kv* kv, const void* kv8, const void* q,
                               const int32_t* idx, int32_t idx_stride, const int32_t* count,
                               float scale, float* out, float* m, float* l, void* workspace,
                               size_t workspace_bytes, dsa_stream_t stream) {
  return quantized_attn(kv, kv8, 8, q, idx, idx_stride, count, scale, out, m, l, workspace,
                        workspace_bytes, stream, "dsa_sparse_decode_attn_kv8");
}

int dsa_quantize_kv4(const dsa_paged_kv* kv, void* kv4, dsa_stream_t stream) {
  return quantize_pool(kv, kv4, 4, stream, "dsa_quantize_kv4");
}

size_t dsa_kv4_bytes(const dsa_paged_kv* kv) { return pool_block_bytes(kv, 136); }

size_t dsa_sparse_decode_attn_kv4_workspace_size(const dsa_paged_kv* kv, int32_t idx_stride) {
  return quantized_attn_workspace(kv, idx_stride);
}

int dsa_sparse_decode_attn_kv4(const dsa_paged_kv* kv, const void* kv4, const void* q,
                               const int32_t* idx, int32_t idx_stride, const int32_t* count,
                               float scale, float* out, float* m, float* l, void* workspace,
                               size_t workspace_bytes, dsa_stream_t stream) {
  return quantized_attn(kv, kv4, 4, q, idx, idx_stride, count, scale, out, m, l, workspace,
                        workspace_bytes, stream, "dsa_sparse_decode_attn_kv4");
}

size_t dsa_calibrate_ema_workspace_size(int32_t steps, int32_t rows, int32_t n, int32_t k) {
  if (steps < 1 || rows < 1 || n < 1 || k < 1) return 16;
  return calib_workspace(steps, rows, n, k).total;
}

int dsa_calibrate_ema(const float* traj, int32_t steps, int32_t rows, int32_t n, int32_t stride,
                      int32_t k, int32_t k_pred, float* H, int32_t* best, void* workspace,
                      size_t workspace_bytes, dsa_stream_t stream) {
  if (steps < 0 || rows < 0 || n < 0) return fail(DSA_ERR_INVALID_ARG, "negative size");
  if (rows == 0) return ok();
  if (steps < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_calibrate_ema: steps must be >= 1");
  if (!traj || !H || !best) return fail(DSA_ERR_INVALID_ARG, "traj/H/best is NULL");
  if (n < 1 || n > stride) return fail(DSA_ERR_INVALID_ARG, "need 1 <= n <= stride");
  if (n > kCalibMaxN) return fail(DSA_ERR_UNSUPPORTED, "n %d > %d", n, kCalibMaxN);
  if (k < 1 || k_pred < 1) return fail(DSA_ERR_INVALID_ARG, "k and k_pred must be >= 1");
  if (k > kMaxListPages || k_pred > kMaxListPages)
    return fail(DSA_ERR_UNSUPPORTED, "k and k_pred must be <= %d", kMaxListPages);
  if (static_cast<long long>(rows) * kCalibPoints > 0x7fffffffLL)
    return fail(DSA_ERR_UNSUPPORTED, "too many rows");
  const size_t need = dsa_calibrate_ema_workspace_size(steps, rows, n, k);
  if (!workspace || workspace_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return fail(DSA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  if (static_cast<long long>(steps) * rows > 0x7fffffffLL)
    return fail(DSA_ERR_UNSUPPORTED, "steps * rows too large");
  cudaError_t e = launch_calib(traj, steps, rows, n, stride, k, k_pred, H, best, workspace,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_calibrate_ema launch");
}

int dsa_merge_partials(const float* partials, int32_t rows, int32_t num_parts, int32_t group,
                       int32_t head_dim, float* out, float* m, float* l, dsa_stream_t stream) {
  if (rows < 0 || num_parts < 0) return fail(DSA_ERR_INVALID_ARG, "negative size");
  if (rows == 0) return ok();
  if (!partials || !out || !m || !l) return fail(DSA_ERR_INVALID_ARG, "NULL pointer");
  if (head_dim != kHeadDim) return fail(DSA_ERR_UNSUPPORTED, "head_dim must be 128");
  if (group < 1 || group > 65535) return fail(DSA_ERR_INVALID_ARG, "bad group");
  MergeArgs mg = {};
  mg.part = partials;
  mg.slots = num_parts;
  mg.rows = rows;
  mg.G = group;
  mg.Hkv = 1;
  mg.Hq = group;
  mg.out = out;
  mg.m = m;
  mg.l = l;
  mg.out_rows_are_heads = 0;
  cudaError_t e = launch_merge(mg, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_merge_partials launch");
}

size_t dsa_sparse_decode_attn_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

int dsa_sparse_decode_attn_noalloc(const dsa_paged_kv* kv, const void* q, const int32_t* idx,
                                   int32_t idx_stride, const int32_t* count, float scale,
                                   float* out, float* m, float* l, int32_t num_splits,
                                   dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!q || !idx || !count || !out || !m || !l)
    return fail(DSA_ERR_INVALID_ARG, "q/idx/count/out/m/l is NULL");
  if (idx_stride < 1) return fail(DSA_ERR_INVALID_ARG, "idx_stride < 1");
  if (!aligned(q, 16)) return fail(DSA_ERR_ALIGNMENT, "q must be 16-byte aligned");
  const int rows = v.B * v.Hkv;
  const int splits = auto_splits(rows, idx_stride, num_splits);
  const size_t need = splits > 1 ? record_bytes(rows, splits, v.G) : 0;
  if (need > kNoAllocScratchBytes)
    return fail(DSA_ERR_UNSUPPORTED,
                "dsa_sparse_decode_attn_noalloc: %d rows x %d splits x %d heads need %zu bytes of "
                "split records, more than its fixed %zu-byte scratch; pass fewer splits or use "
                "dsa_sparse_decode_attn with a workspace",
                rows, splits, v.G, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if (need > 0 && (rc = noalloc_scratch(&scratch))) return rc;
  CUtensorMap tk, tv;
  if ((rc = pool_map(kv->k_pages, kv, &tk)) || (rc = pool_map(kv->v_pages, kv, &tv))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AttnArgs a = {};
  a.kv = v;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.scale_log2 = scale_log2(scale);
  a.idx = idx;
  a.idx_stride = idx_stride;
  a.count = count;
  a.num_splits = splits;
  a.stages = attn_stages(v.p, (idx_stride + splits - 1) / splits);
  a.out = out;
  a.m = m;
  a.l = l;
  // every split slot of every row is written before the merge reads it, so the scratch needs
  // no clearing between calls
  if (splits > 1) {
    a.part = static_cast<float*>(scratch);
    a.part_slots = splits;
  }
  cudaError_t e = launch_attn(LIST_SELECTED, tk, tv, a, splits, s);
  if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_decode_attn_noalloc launch");
  if (splits > 1) {
    MergeArgs mg = {};
    mg.part = static_cast<const float*>(scratch);
    mg.slots = splits;
    mg.rows = rows;
    mg.G = v.G;
    mg.Hkv = v.Hkv;
    mg.Hq = v.Hq;
    mg.streaming = v.streaming;
    mg.out = out;
    mg.m = m;
    mg.l = l;
    mg.out_rows_are_heads = 1;
    e = launch_merge(mg, s);
    if (e != cudaSuccess) return cuda_fail(e, "dsa_sparse_decode_attn_noalloc merge");
  }
  return ok();
}

size_t dsa_prr_step_workspace_size(const dsa_paged_kv* kv) {
  if (!kv || kv->batch <= 0 || kv->num_kv_heads <= 0 || kv->max_pages_per_seq <= 0) return 0;
  return prr_step_workspace_bytes(kv->batch * kv->num_kv_heads, kv->max_pages_per_seq);
}

size_t dsa_prr_step_counter_bytes(const dsa_paged_kv* kv) {
  if (!kv || kv->batch <= 0 || kv->num_kv_heads <= 0) return 0;
  return prr_step_counter_bytes(kv->batch * kv->num_kv_heads);
}

int dsa_prr_step(const dsa_paged_kv* kv, const dsa_prr_step_args* args, void* workspace,
                 size_t workspace_bytes, dsa_stream_t stream) {
  KvView v;
  int rc = check_kv(kv, 2, &v);
  if (rc) return rc;
  if (!args) return fail(DSA_ERR_INVALID_ARG, "dsa_prr_step: args is NULL");
  const dsa_prr_step_args& x = *args;
  if (!x.q || !x.meta || !x.scores || !x.ell || !x.trend || !x.spec_idx || !x.spec_count ||
      !x.page_partials || !x.idx || !x.count || !x.next_idx || !x.next_count || !x.out || !x.m ||
      !x.l)
    return fail(DSA_ERR_INVALID_ARG, "dsa_prr_step: a required pointer is NULL");
  if (v.streaming != nullptr)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_prr_step: streaming heads are not supported");
  if (x.k < 1 || x.k_pred < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_prr_step: k and k_pred >= 1");
  if (x.stride < v.max_pages || x.stride > kMaxSelectN)
    return fail(DSA_ERR_INVALID_ARG, "dsa_prr_step: stride must be in [max_pages_per_seq, %d]",
                kMaxSelectN);
  if (x.k > kMaxListPages || x.k_pred > kMaxListPages)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_prr_step: k and k_pred must be <= %d", kMaxListPages);
  if (x.next_idx == x.spec_idx || x.next_count == x.spec_count)
    return fail(DSA_ERR_INVALID_ARG, "dsa_prr_step: next_idx/next_count must not alias P_t");
  if (!aligned(x.q, 16) || !aligned(x.meta, 16) || !aligned(x.page_partials, 16))
    return fail(DSA_ERR_ALIGNMENT, "dsa_prr_step: q, meta and page_partials must be 16-byte aligned");
  const size_t ws_need = prr_step_workspace_bytes(v.B * v.Hkv, v.max_pages);
  if (!workspace || workspace_bytes < ws_need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes needed", ws_need);
  if (!aligned(workspace, 16)) return fail(DSA_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  if (prr_step_smem_bytes(v.p, x.stride, x.k_pred) > kPrrSmemLimit)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_prr_step: shape needs too much shared memory");
  CUtensorMap tk, tv;
  if ((rc = pool_map(kv->k_pages, kv, &tk)) || (rc = pool_map(kv->v_pages, kv, &tv))) return rc;
  PrrStepArgs a = {};
  a.kv = v;
  a.kpool = static_cast<const __nv_bfloat16*>(kv->k_pages);
  a.vpool = static_cast<const __nv_bfloat16*>(kv->v_pages);
  a.q = static_cast<const __nv_bfloat16*>(x.q);
  a.meta = static_cast<const uint8_t*>(x.meta);
  a.scores = x.scores;
  a.stride = x.stride;
  a.ell = x.ell;
  a.trend = x.trend;
  a.alpha = x.alpha;
  a.beta = x.beta;
  a.gamma = x.gamma;
  a.pred = x.pred;
  a.spec_idx = x.spec_idx;
  a.spec_count = x.spec_count;
  a.k_pred = x.k_pred;
  a.partials = x.page_partials;
  a.idx = x.idx;
  a.count = x.count;
  a.k = x.k;
  a.next_idx = x.next_idx;
  a.next_count = x.next_count;
  a.superset = x.superset != 0;
  a.scale_log2 = scale_log2(x.scale);
  a.out = x.out;
  a.m = x.m;
  a.l = x.l;
  const cudaError_t e = launch_prr_step(tk, tv, a, workspace, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "dsa_prr_step launch");
}

}  // extern "C"
