// One whole PRR decode step (t >= 1) in a single launch of one CTA per SM ("Predict, Reuse, and Repair"
// §3: speculation over the predicted set P_t, the true selection A_t, the predictor update, repair
// of the missed pages and the merge), organised so that no CTA ever waits for the whole grid.
//
// Roles.  With few (row, query head) tasks (at most a quarter of the grid), the first CTAs only run
// tasks and the others (the workers) score; a task CTA's compute warps take its task's first steps
// (the P_t list, the bitmaps, the row's workers) while its eighth warp attends its pages of P_t.
// Otherwise every CTA is a worker first and then takes tasks round robin.
//   scoring  each worker scores an equal share of the (row, page) slots with the scoring kernel's
//            arithmetic (every page-table entry, length, EMA state and query load of a round in
//            flight at once, then the metadata records), updates the EMA state of those pages at
//            once (no other CTA reads their old state), and counts the row's scored pages up by
//            its share (one counter per row).  Pages scoring at or above the row's hint (a key
//            the previous call left, see below) go to the worker's candidate line for the row as
//            they are found, so that they are out before the count;
//   items    the pages of P_t are spread over every CTA's eighth warp, which issues their TMA
//            loads through the CTA's ring, attends each page (all of its 16-token tiles, the whole
//            query group as the m16 tile of the tensor-core products) while the other warps score,
//            and writes the page's record straight from its registers, counted per row;
//   tasks    per (row, query head), once the row is scored: A_t.  When the covering workers listed
//            at least k candidates (and none overflowed its line), the row's k best are among
//            them and only the list is ranked; the k best are marked in a bitmap and read out in
//            ascending order.  Otherwise the row's scores (L2, one batch of loads) are ranked with
//            T0, the k-th largest score over P_t's pages, as the lower bound of A_t's cut-off, or
//            every page when that does not hold.  The first head's task publishes A_t and the next
//            hint: the key of rank 1.5k when the list reached it, else the score where rank 1.75k
//            would stand if the top scores' log-rank is linear in the score.  Any hint value is
//            safe; it only decides how often the list is usable.  The missed pages A_t \ P_t go
//            through the ring (one warp per page, looked up in a bitmap of P_t), and the task
//            merges them with the records of A_t ∩ P_t (all of P_t in superset mode).  Per row,
//            one more task ranks P_{t+1} from the new predictions with T0's counterpart (the
//            k_pred-th largest prediction over P_t).
// Each wait is on a per-row counter that only work done before any wait advances, so every wait
// ends; all are bounded (DSA_STATUS_TIMEOUT after 2 s).  Every CTA arrives at an exit count after
// its last wait (a merge task's eighth warp in mid-task, the other CTAs on their way out); the
// last to arrive sets the counters back to zero.
#include "attn_core.cuh"
#include "internal.h"
#include "score_core.cuh"
#include "select.cuh"

namespace dsa {
#ifdef DSA_TIMELINE
__device__ unsigned long long g_trace_prr[kTraceCtas * 2 * kTraceSlots];
#endif
namespace {

// 8 warps (two per SM sub-partition) leave every thread up to 255 registers
constexpr int kW = 7;                      // compute warps
constexpr int kThreads = (kW + 1) * 32;    // + one TMA issue warp
constexpr int kWarps = kThreads / 32;
constexpr int kCT = kW * 32;               // compute threads
constexpr int kGroups = kCT / 8;           // scoring record groups of 8 lanes
constexpr int kRecGroup = 5;               // records per group per scoring round
constexpr int kRound = kGroups * kRecGroup;
constexpr int kPredMax = kPrrPredMax;      // bound of k and k_pred
constexpr int kMaxStages = 3;              // TMA ring depth
constexpr int kWs = kHeadDim + 4;          // a warp's merge state: m, l, -, -, O[128]
constexpr int kRoundRecs = 10;             // records a warp loads at once in the merge
constexpr int kQTile = 16 * kQStride;      // bf16 elements of one warp's query tile
constexpr int kBitsMax = kTopkMaxN / 2;    // longest row the A_t pass keeps two bitmaps for


// ------------------------------------------------------------------------------ shared memory

struct SLayout {
  uint32_t stage_off, q_off;  // the ring and the warps' query tiles (items, missed pages)
  uint32_t keys_off;          // a row's keys (selection; shares the ring's space)
  uint32_t rec_off;           // P_t's records of one query head (tasks; optional)
  uint32_t qbar_off, pl_off, pk_off, sa_off, list_off, parts_off, ws_off;
  uint32_t total;
};

__host__ __device__ inline uint32_t up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SLayout slayout(int page, int n, int k_pred, int S, bool rec_smem) {
  SLayout L;
  L.stage_off = 0;
  L.q_off = S * 512u * page;
  const uint32_t ring_end = L.q_off + kWarps * kQTile * 2u;  // a query tile per warp
  L.keys_off = 0;
  const uint32_t keys_end = 16u * ((n + 3) / 4);  // zero-padded to whole 4-key groups
  L.rec_off = up(ring_end > keys_end ? ring_end : keys_end, 16);
  L.qbar_off = up(L.rec_off + (rec_smem ? 4u * kRecordFloats * k_pred : 0u), 16);
  L.pl_off = L.qbar_off + kHeadDim * 4u;
  L.pk_off = L.pl_off + kPredMax * 4u;
  L.sa_off = L.pk_off + kPredMax * 4u;
  L.list_off = L.sa_off + kPredMax * 4u;
  L.parts_off = L.list_off + kPredMax * 4u;
  L.ws_off = L.parts_off + kPredMax * 4u;
  L.total = L.ws_off + kWarps * kWs * 4u + 1024u;  // + alignment slack
  return L;
}

// ------------------------------------------------------------------------------ workspace

constexpr int kMaxWorkers = 160;  // worker CTAs the candidate lists have room for
constexpr int kWorkerSlots = 16;  // one 128-byte line per (row, worker): up to 15 candidates, then
constexpr int kWorkerCand = kWorkerSlots - 1;  // a slot that is nonzero when more were found

struct WsLayout {
  size_t exit_off, done_off, sdone_off, counters, hint_off, cand_off, pred_off, total;
};

inline WsLayout ws_layout(int rows, int max_pages) {
  auto a16 = [](size_t x) { return (x + 15) & ~static_cast<size_t>(15); };
  const size_t cnt = a16(4 * static_cast<size_t>(rows));
  WsLayout w;
  w.exit_off = 0;
  w.done_off = 16;
  w.sdone_off = w.done_off + cnt;
  w.counters = w.sdone_off + cnt;
  w.hint_off = a16(w.counters);
  w.cand_off = w.hint_off + cnt;
  w.pred_off = w.cand_off + 8 * static_cast<size_t>(rows) * kMaxWorkers * kWorkerSlots;
  w.total = w.pred_off + 4 * static_cast<size_t>(rows) * max_pages;
  return w;
}

struct Ws {
  unsigned* exit;    // CTAs finished
  unsigned* done;    // [rows] pages scored (and their EMA state updated)
  unsigned* sdone;   // [rows] records of P_t written
  uint32_t* hint;    // [rows] key the workers list candidates from (0: none); kept across steps
  unsigned long long* cand;  // [rows][kMaxWorkers][kWorkerSlots] a worker's candidates as (key,
                             // position) rank values, 0 past them, the last slot nonzero when it
                             // found more (a worker clears its line each call)
  float* pred;       // [rows][max_pages] the new predictions
};

// (key, position) as one 64-bit value ordered by key, then by the lower position.
DSA_DEV unsigned long long rank_value_of(uint32_t key, int pos) {
  return (static_cast<unsigned long long>(key) << 32) | (0xffffffffu - static_cast<uint32_t>(pos));
}
DSA_DEV int rank_pos_of(unsigned long long v) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(v));
}

// ------------------------------------------------------------------------------ waits

DSA_DEV unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One thread: waits until *ctr reaches target (compared as a sequence number).  Each poll is one
// L2 round trip and there is no sleep between polls, so the count is seen complete about one
// round trip after its last increment; one thread per CTA polls.  Bounded: gives up after
// kWaitLimitNs, raising DSA_STATUS_TIMEOUT and the CTA's abort flag.
DSA_DEV void wait_count(const unsigned* ctr, unsigned target, volatile int* abort,
                        int32_t* status) {
  if (*abort || static_cast<int>(ld_acquire(ctr) - target) >= 0) return;
  const unsigned long long t0 = global_timer_ns();
  while (static_cast<int>(ld_acquire(ctr) - target) < 0) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      raise_status(status, DSA_STATUS_TIMEOUT);
      return;
    }
  }
}

// Makes the writes so far of the threads that just passed a barrier with this one visible, then
// advances the counter.
DSA_DEV void publish_add(unsigned* ctr, unsigned v) {
  __threadfence();
  atomicAdd(ctr, v);
}

struct PrrArgs {
  KvView kv;
  const __nv_bfloat16* q;
  const uint8_t* meta;
  float* scores;
  int stride;  // score / EMA row stride = pages per row
  float* ell;
  float* trend;
  float alpha, beta, gamma;
  float* pred;
  const int32_t* spec_idx;
  const int32_t* spec_count;
  int k_pred;
  float* partials;  // [rows][k_pred][G][kRecordFloats]
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
  Ws ws;
  int stages;
  int rec_smem;  // P_t's records of a task's query head staged in shared memory
};

__global__ void __launch_bounds__(kThreads, 1)
    prr_step_kernel(const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const PrrArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  __shared__ __align__(16) SelectAnyScratch<kThreads> sel;  // candidate keys are read as uint4
  // the ring's mbarriers ([S] full, [S] empty) and stage descriptors
  __shared__ __align__(8) uint64_t bars[2 * kMaxStages];
  __shared__ int s_ctl[2 * kMaxStages];
  __shared__ int s_abort, s_issued, s_red[4];
  __shared__ unsigned s_t0, s_hint, s_kmid, s_klow;
  __shared__ int s_wlo, s_whi;  // the workers whose shares meet a task's row
  __shared__ int s_ccnt;  // a worker's candidates of the current segment
  __shared__ int s_cntp;  // |P_t| of a task prepared during the worker phase
  const KvView& kv = a.kv;
  const Ws& W = a.ws;
  const int page = kv.p, G = kv.G, tiles = page / 16, S = a.stages;
  const int rows = kv.B * kv.Hkv, n = a.stride, kp = a.k_pred;
  const SLayout lay = slayout(page, n, kp, S, a.rec_smem != 0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t stage_bytes = 512u * page;
  const int grid = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);

  // roles
  const int n_tasks = rows * G + rows;
  const bool split = 4 * n_tasks <= grid;
  const int work_base = split ? n_tasks : 0, workers = grid - work_base;
  const int wk = cta - work_base;  // rank among the workers (negative: a task CTA)
  // a worker's equal share [s_beg, s_end) of the (row, page) slots.  The items of P_t (the
  // speculative pages) are spread over every CTA's TMA issue warp, which attends them while the
  // compute warps score: this CTA's items are cta + j * grid for j < my_items.
  const long long T = static_cast<long long>(rows) * n;
  const long long s_beg = wk < 0 ? 0 : static_cast<long long>(wk) * T / workers;
  const long long s_end = wk < 0 ? 0 : static_cast<long long>(wk + 1) * T / workers;
  const int n_items = rows * kp;
  const int my_items = cta < n_items ? (n_items - 1 - cta) / grid + 1 : 0;

  // a merge task's first steps need neither the row's scores nor the ring (compute warps): its
  // bitmaps cleared and P_t's positions (in pl) marked, the workers whose shares meet its row
  // found.  A barrier of the compute warps must follow before these are read.
  TopkScratch& ts = sel.small;
  int32_t* pl = reinterpret_cast<int32_t*>(smem + lay.pl_off);  // P_t's positions
  auto merge_prep = [&](int row, int cntP) {
    const int nwords = (n + 31) >> 5;
    uint32_t* abits = ts.bits;
    uint32_t* pbits = ts.bits + kBitsMax / 32;
    if (n <= kBitsMax)
      for (int w = tid; w < nwords; w += kCT) abits[w] = pbits[w] = 0u;
    if (tid == 0) {
      s_hint = 0u;
      ts.n_cand = 0;
    }
    if (tid == 32) {
      // the workers whose shares [w T / workers, (w + 1) T / workers) meet [r0, r1): from the
      // one holding slot r0 to the one holding slot r1 - 1
      const long long r0 = static_cast<long long>(row) * n, r1 = r0 + n;
      auto holder = [&](long long x) {
        int w = static_cast<int>(min(static_cast<long long>(workers - 1), x * workers / T));
        while (w > 0 && static_cast<long long>(w) * T / workers > x) --w;
        while (w + 1 < workers && static_cast<long long>(w + 1) * T / workers <= x) ++w;
        return w;
      };
      s_wlo = holder(r0);
      s_whi = holder(r1 - 1);
    }
    named_barrier(1, kCT);
    if (n <= kBitsMax)
      for (int i = tid; i < cntP; i += kCT)
        if (pl[i] >= 0 && pl[i] < n) atomicOr(&pbits[pl[i] >> 5], 1u << (pl[i] & 31));
  };
  // in split mode a merge-task CTA has one task, known now: its compute warps, idle while the issue
  // warp attends the CTA's page of P_t, take the task's first steps meanwhile
  const bool pre = split && cta < rows * G;

  volatile int* stage_ok = s_ctl;  // -1 nothing, 0 empty part, 1 page loaded
  volatile int* stage_pos = s_ctl + S;
  __nv_bfloat16* sQw = reinterpret_cast<__nv_bfloat16*>(smem + lay.q_off) + warp * kQTile;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[S + s]), 1);
    }
    fence_mbar_init();
    s_abort = 0;
    s_issued = 0;
  }
  // everything above touches shared memory and the arguments only; from here on global memory
  // written by earlier kernels is read
  launch_dependents();
  grid_dependency_wait();
  __syncthreads();
  DSA_TRACE_BEGIN();

  // ---- the TMA ring, shared by the speculative pages (workers) and the missed pages (tasks):
  // ring position j uses stage j % S with phase parity (j / S) & 1 and is consumed by warp j % S,
  // so each stage's phases are waited for in order by one warp.
  // issue warp, lane 0: item j; `has` false completes the stage with nothing to attend
  auto issue = [&](int j, int row, int pos, bool has, int npos) -> bool {
    const int s = j % S, u = j / S;
    if (u > 0 && !mbar_wait(smem_u32(&bars[S + s]), (u - 1) & 1, abort_flag, kv.status))
      return false;
    int okv = -1, phys = 0;
    if (has) okv = lookup_page(kv, row / kv.Hkv, pos, npos, &phys) ? 1 : 0;
    const uint32_t full = smem_u32(&bars[s]);
    stage_ok[s] = okv;
    stage_pos[s] = pos;
    if (okv == 1) {
      const uint32_t dst = smem_base + s * stage_bytes;
      const int row0 = (phys * kv.Hkv + row % kv.Hkv) * page;
      mbar_arrive_expect_tx(full, stage_bytes);
      tma_load_page(dst, &tmK, row0, full);
      tma_load_page(dst + 2 * page * 128, &tmV, row0, full);
    } else {
      mbar_arrive(full);
    }
    *reinterpret_cast<volatile int*>(&s_issued) = j + 1;
    return true;
  };
  // one warp: the query rows of a row's group into the warp's tile (rows past G are zero), then
  // their A fragments
  auto warp_q = [&](int row, uint32_t (&qa)[8][4]) {
    const int b = row / kv.Hkv, h = row % kv.Hkv;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int piece = lane + 32 * i, r = piece >> 4, c = piece & 15;
      __nv_bfloat16* dst = sQw + r * kQStride + c * 8;
      if (r < G)
        cp_async16(smem_u32(dst),
                   a.q + (static_cast<size_t>(b) * kv.Hq + h * G + r) * kHeadDim + c * 8);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_wait_all();
    __syncwarp();
    load_q_frags(sQw, qa);
    __syncwarp();
  };
  // one warp: attention of the query group over the page of ring item j (tokens < L), folded into
  // st.  Returns the stage's state (-1 nothing, 0 no page, 1 attended) or -2 after a timeout.
  auto attend_item = [&](int j, int L, const uint32_t (&qa)[8][4], WarpSoftmaxState& st) -> int {
    const int s = j % S;
    const bool got = mbar_wait(smem_u32(&bars[s]), (j / S) & 1, abort_flag, kv.status);
    const int okv = got ? stage_ok[s] : -1;
    const int pos = stage_pos[s];
    if (okv == 1) {
      const uint32_t kb = smem_base + s * stage_bytes;
      const uint32_t vb = kb + 2 * page * 128;
      bool wrote = false;
      for (int t = 0; t < tiles; ++t) {
        const bool in = pos * page + t * 16 + (lane & 15) < L;
        const uint32_t vm = __ballot_sync(0xffffffffu, in) & 0xffffu;
        if (vm == 0u) continue;
        if (vm != 0xffffu)
          wrote |= zero_invalid_v_rows(vm, smem + s * stage_bytes + 2 * page * 128, page, t * 16);
        float sc[2][4];
        tile_scores(qa, kb, page, t * 16, sc);
        tile_softmax_pv(st, sc, a.scale_log2, vm, vb, page, t * 16);
      }
      if (wrote) fence_proxy_async_smem();
    }
    __syncwarp();
    if (got && lane == 0) mbar_arrive(smem_u32(&bars[S + s]));
    return got ? okv : -2;
  };
  // waits (bounded) for this CTA's page loads still in flight: after a timeout
  auto drain = [&]() {
    if (tid == 0) {
      const int n_iss = *reinterpret_cast<volatile int*>(&s_issued);
      for (int j = max(0, n_iss - S); j < n_iss; ++j) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&bars[j % S]), (j / S) & 1))
          if (global_timer_ns() - t0 > 50000000ull) break;
      }
    }
  };

  if (warp == kW) {
    // ================================================================ TMA issue warp
    // this CTA's items of P_t: lane 0 issues up to S of them at once, the warp attends each into
    // its page records (published per item), and each stage it frees takes the item S later
    auto issue_item = [&](int j) -> bool {
      const int it = cta + j * grid;
      const int row = it / kp, slot = it - row * kp;
      // the three loads go out together
      const int cnt = a.spec_count[row];
      const int pos = a.spec_idx[static_cast<size_t>(row) * kp + slot];
      const int npos = (request_len(kv, row / kv.Hkv) + page - 1) / page;
      return issue(j, row, pos, slot < min(max(cnt, 0), kp), npos);
    };
    bool ok = true;
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      for (int j = 0; j < my_items && j < S && ok; ++j) ok = issue_item(j);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
    for (int j = 0; j < my_items && ok; ++j) {
      const int it = cta + j * grid;
      const int row = it / kp, pslot = it - row * kp;
      uint32_t qa[8][4];
      warp_q(row, qa);
      WarpSoftmaxState st;
      state_init(st);
      const int okv = attend_item(j, request_len(kv, row / kv.Hkv), qa, st);
      if (okv == -2) break;
      if (lane == 0 && j + S < my_items) ok = issue_item(j + S);  // the stage just freed
      ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
      if (okv < 0) continue;
      state_finish(st);
      float* rec0 = a.partials + (static_cast<size_t>(row) * kp + pslot) * G * kRecordFloats;
      // lane holds rows lane / 4 and lane / 4 + 8, dims 8 jj + 2 (lane % 4) + {0, 1}
      const int r0 = lane >> 2, c0 = (lane & 3) * 2;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = r0 + 8 * half;
        if (r >= G) continue;
        float* rec = rec0 + r * kRecordFloats;
        const float lr = okv == 1 ? st.l[half] : 0.f;
        const float inv = lr > 0.f ? 1.f / lr : 0.f;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          *reinterpret_cast<float2*>(rec + jj * 8 + c0) =
              make_float2(st.o[jj][2 * half] * inv, st.o[jj][2 * half + 1] * inv);
        if ((lane & 3) == 0)
          *reinterpret_cast<float4*>(rec + 128) =
              make_float4(lr > 0.f ? st.m[half] * kLn2 : -INFINITY, lr, 0.f, 0.f);
      }
      __syncwarp();
      if (lane == 0) publish_add(W.sdone + row, 1u);
    }
    __syncwarp();
  } else {
    // ================================================================ compute warps
    float* qbar = reinterpret_cast<float*>(smem + lay.qbar_off);
    const int gl = lane & 7, gid = tid >> 3;
    // ---- scoring of the share, one segment (the part inside one row) at a time
    for (long long seg = s_beg; seg < s_end;) {
      const int row = static_cast<int>(seg / n);
      const int j0 = static_cast<int>(seg - static_cast<long long>(row) * n);
      const int j1 = static_cast<int>(min(s_end - static_cast<long long>(row) * n,
                                          static_cast<long long>(n)));
      seg = static_cast<long long>(row) * n + j1;
      const int b = row / kv.Hkv, h = row % kv.Hkv;
      const int32_t* table = kv.page_table + static_cast<size_t>(b) * kv.max_pages;
      float* outs = a.scores + static_cast<size_t>(row) * n;
      float* ell_r = a.ell + static_cast<size_t>(row) * n;
      float* v_r = a.trend + static_cast<size_t>(row) * n;
      float* pred_r = a.pred ? a.pred + static_cast<size_t>(row) * n : nullptr;
      float* wpred_r = W.pred + static_cast<size_t>(row) * kv.max_pages;
      // pages scoring at or above the row's hint (0: none) are A_t candidates, stored as they are
      // found into this worker's slots of the row, cleared first (the merge tasks know which
      // workers cover a row); all of it goes out well before the scores are published
      const bool lists = wk < kMaxWorkers;
      const uint32_t hint = lists ? W.hint[row] : 0u;
      unsigned long long* cand_w =
          W.cand + (static_cast<size_t>(row) * kMaxWorkers + max(wk, 0)) * kWorkerSlots;
      if (lists && tid < kWorkerSlots) cand_w[tid] = 0ull;
      if (tid == 0) s_ccnt = 0;
      named_barrier(1, kCT);  // the previous segment's query is no longer read
      int nl = 0;
      for (int jb = j0; jb < j1; jb += kRound) {
        // indices are clamped rather than guarded, so that every load of the round issues at once
        int ph[kRecGroup];
        float lo[kRecGroup], vo[kRecGroup];
#pragma unroll
        for (int i = 0; i < kRecGroup; ++i) {
          const int jj = jb + gid + kGroups * i;
          const int jc = min(jj, j1 - 1);
          const int phv = table[min(jc, kv.max_pages - 1)];
          const float lv = ell_r[jc], vv = v_r[jc];
          ph[i] = jj < j1 && jj < kv.max_pages ? phv : -1;
          lo[i] = jj < j1 ? lv : 0.f;
          vo[i] = jj < j1 ? vv : 0.f;
        }
        if (jb == j0) {
          nl = (request_len(kv, b) + page - 1) / page;
          // the representative query: the mean of the group's rows (G <= 16: every load in
          // flight, then the sum in row order, as the scoring kernel rounds it)
          if (tid < kHeadDim) {
            const __nv_bfloat16* qg = a.q + (static_cast<size_t>(b) * kv.Hq + h * G) * kHeadDim;
            __nv_bfloat16 qr[kMaxGroup];
#pragma unroll
            for (int r = 0; r < kMaxGroup; ++r)
              qr[r] = r < G ? qg[r * kHeadDim + tid] : __float2bfloat16(0.f);
            float qs = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxGroup; ++r)
              if (r < G) qs += __bfloat162float(qr[r]);
            qbar[tid] = qs / static_cast<float>(G);
          }
          named_barrier(1, kCT);
          DSA_STAMP(1);  // worker: the first segment's table, state and query loaded
        }
        float qv[16];
        group_query_dims(qbar, gl, qv);
        uint4 rc[kRecGroup][4];
        bool okr[kRecGroup], bad = false;
#pragma unroll
        for (int i = 0; i < kRecGroup; ++i) {
          const int jj = jb + gid + kGroups * i;
          const bool in = jj < j1 && jj < nl;
          okr[i] = in && ph[i] >= 0 && ph[i] < kv.num_phys;
          bad |= in && !okr[i];
          // a slot without a page loads page 0's record and discards it
          load_record(a.meta, static_cast<size_t>(okr[i] ? ph[i] : 0) * kv.Hkv + h, gl, rc[i]);
        }
        if (gl == 0 && bad) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
        DSA_STAMP(16);  // worker: the round's record loads issued
#pragma unroll
        for (int i = 0; i < kRecGroup; ++i) {
          const int jj = jb + gid + kGroups * i;
          const float sc = group_sum(okr[i] ? record_partial<DSA_META_MINMAX>(rc[i], qv) : 0.f);
          if (gl == 0 && jj < j1) {
            const float is = okr[i] ? sc : -INFINITY;
            outs[jj] = is;
            const uint32_t key = score_key(is);
            if (hint != 0u && key >= hint) {
              const int at = atomicAdd(&s_ccnt, 1);
              cand_w[min(at, kWorkerCand)] = at < kWorkerCand ? rank_value_of(key, jj) : 1ull;
            }
            float l_new, v_new;
            ema_step(is, lo[i], vo[i], DSA_EMA_UPDATE, a.alpha, a.beta, l_new, v_new);
            const float pr = ema_predict(l_new, v_new, a.gamma);
            ell_r[jj] = l_new;
            v_r[jj] = v_new;
            if (pred_r) pred_r[jj] = pr;
            if (jj < kv.max_pages) wpred_r[jj] = pr;
          }
        }
        DSA_STAMP(17);  // worker: thread 0's scores and EMA state of the round written
      }
      named_barrier(1, kCT);
      DSA_STAMP(18);  // worker: the segment's rounds done (barrier)
      if (tid == 0) publish_add(W.done + row, static_cast<unsigned>(j1 - j0));
    }
    DSA_STAMP(2);  // worker: its share scored and published

    DSA_STAMP(3);  // the compute warps' part is over (thread 0)
    if (pre) {
      const int row = cta / G;
      const int cntP = min(max(a.spec_count[row], 0), kp);
      for (int i = tid; i < cntP; i += kCT) pl[i] = a.spec_idx[static_cast<size_t>(row) * kp + i];
      if (tid == 0) s_cntp = cntP;
      named_barrier(1, kCT);  // pl written
      merge_prep(row, cntP);
    }
  }
  __syncthreads();
  DSA_STAMP(4);  // the CTA's worker part is over
  if (*abort_flag) {
    drain();
    return;
  }

  // ================================================================ tasks
  // (row, query head) merges first, then one P_{t+1} selection per row.  In a merge the seven
  // compute warps select A_t while the TMA issue warp brings the speculative records of the task's
  // query head on chip.
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + lay.keys_off);  // a row's keys
  float* srec = reinterpret_cast<float*>(smem + lay.rec_off);  // P_t's records of one head
  uint32_t* pk = reinterpret_cast<uint32_t*>(smem + lay.pk_off);  // their keys
  int32_t* sA = reinterpret_cast<int32_t*>(smem + lay.sa_off);
  int32_t* mlist = reinterpret_cast<int32_t*>(smem + lay.list_off);  // missed positions
  int32_t* parts = reinterpret_cast<int32_t*>(smem + lay.parts_off);
  float* wst = reinterpret_cast<float*>(smem + lay.ws_off);  // [warp][m, l, -, -, O[128]]
  const unsigned below = (1u << lane) - 1u;
  int ring = my_items;  // next ring position (the same in every thread)

  // keys[j] = key of src[j] for j < n_src, 0 for n_src <= j < n rounded up to 4 (src: an fp32 row
  // of other CTAs' writes, read through L2 with all of a thread's loads in flight); compute warps
  auto load_keys = [&](const float* src, int n_src) {
    if ((n_src & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      const int n4 = n_src >> 2;
      for (int i0 = tid; i0 < n4; i0 += 8 * kCT) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + u * kCT < n4) v[u] = __ldcg(reinterpret_cast<const float4*>(src) + i0 + u * kCT);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + u * kCT < n4)
            *reinterpret_cast<uint4*>(keys + 4 * (i0 + u * kCT)) = make_uint4(
                score_key(v[u].x), score_key(v[u].y), score_key(v[u].z), score_key(v[u].w));
      }
    } else {
      for (int j0 = tid; j0 < n_src; j0 += 8 * kCT) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = j0 + u * kCT < n_src ? __ldcg(src + j0 + u * kCT) : -INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (j0 + u * kCT < n_src) keys[j0 + u * kCT] = score_key(v[u]);
      }
    }
    for (int j = n_src + tid; j < ((n + 3) & ~3); j += kCT) keys[j] = 0u;
  };
  // Rank of key[i] among key[0, m) by (key descending, position ascending): the keys before i
  // that are >= it plus the keys after i that are > it.  key is 16-byte aligned and padded with
  // zeros to a multiple of 4 (a zero key ranks after every other).
  auto rank_of = [&](const uint32_t* key, int m, int i) -> int {
    const uint32_t ki = key[i];
    const uint4* k4 = reinterpret_cast<const uint4*>(key);
    int r = 0;
    for (int q4 = 0; q4 < ((m + 3) >> 2); ++q4) {
      const uint4 v = k4[q4];
      const int q = 4 * q4;
      r += (q + 0 < i ? v.x >= ki : v.x > ki) + (q + 1 < i ? v.y >= ki : v.y > ki) +
           (q + 2 < i ? v.z >= ki : v.z > ki) + (q + 3 < i ? v.w >= ki : v.w > ki);
    }
    return r;
  };
  // Compute warps: top-kk of the row's keys (keys[0, n), valid = != 0) into out[0, kk) in
  // ascending index order, -1 past the count; returns the count.  The kk-th largest key over P_t's
  // pages (pl[0, cntP)) bounds the kk-th largest of the row from below, so only the C keys at or
  // above it are ranked.  Returns -1 (nothing written) when there is no bound or C > kTopkMaxCand:
  // the whole block then ranks every key.
  auto select_fast = [&](int kk, int cntP, int32_t* out) -> int {
    const int cnt4 = (cntP + 3) & ~3;
    for (int i = tid; i < cnt4; i += kCT) {
      const int pos = i < cntP ? pl[i] : -1;
      pk[i] = pos >= 0 && pos < n ? keys[pos] : 0u;
    }
    if (tid == 0) s_t0 = 0u;
    named_barrier(1, kCT);
    // the bound: P_t's key of rank kk - 1 (kk keys of P_t are >= it)
    for (int i = tid; i < cntP; i += kCT)
      if (pk[i] != 0u && rank_of(pk, cntP, i) == kk - 1) s_t0 = pk[i];
    named_barrier(1, kCT);
    const uint32_t t0 = s_t0;
    if (t0 == 0u) return -1;
    // the keys >= t0 in index order: thread t takes the contiguous 4-key groups of chunk t
    const int n4 = (n + 3) >> 2;
    const int per = (n4 + kCT - 1) / kCT;
    const int g0 = min(n4, tid * per), g1 = min(n4, g0 + per);
    const uint4* k4 = reinterpret_cast<const uint4*>(keys);
    int c = 0;
    for (int gi = g0; gi < g1; ++gi) {
      const uint4 v = k4[gi];
      c += (v.x >= t0) + (v.y >= t0) + (v.z >= t0) + (v.w >= t0);
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) ts.wcnt[warp] = incl;
    named_barrier(1, kCT);
    int C = 0, at = incl - c;
    for (int w = 0; w < kW; ++w) {
      const int wc = ts.wcnt[w];
      if (w < warp) at += wc;
      C += wc;
    }
    if (C > kTopkMaxCand) return -1;
    for (int gi = g0; gi < g1 && c > 0; ++gi) {
      const uint4 v = k4[gi];
      const uint32_t kq[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (kq[e] >= t0) {
          ts.ckey[at] = kq[e];
          ts.cidx[at] = 4 * gi + e;
          ++at;
        }
    }
    for (int i = C + tid; i < ((C + 3) & ~3); i += kCT) ts.ckey[i] = 0u;
    named_barrier(1, kCT);
    // candidate i is among the kk best when fewer than kk rank ahead of it (they are in index
    // order, so ties go to the lower index); its place is the number of selected ones before it
    int o_base = 0;
    for (int i0 = 0; i0 < C; i0 += kCT) {
      const int i = i0 + tid;
      const bool take = i < C && rank_of(ts.ckey, C, i) < kk;
      const unsigned bal = __ballot_sync(0xffffffffu, take);
      if (lane == 0) ts.wcnt[warp] = __popc(bal);
      named_barrier(1, kCT);
      int before = o_base, round = 0;
      for (int w = 0; w < kW; ++w) {
        const int wc = ts.wcnt[w];
        if (w < warp) before += wc;
        round += wc;
      }
      if (take) out[before + __popc(bal & below)] = ts.cidx[i];
      o_base += round;
      named_barrier(1, kCT);
    }
    const int total = min(C, kk);
    for (int i = total + tid; i < kk; i += kCT) out[i] = -1;
    fence_proxy_async_smem();  // the keys' space is the ring's, which TMA writes next
    return total;
  };
  // The whole block: top-kk of every key of the row (the keys are still in place)
  auto select_all = [&](int kk, int32_t* out) -> int {
    KeyStats st;
    for (int j = tid; j < n; j += kThreads) st.add(keys[j]);
    const int total = select_topk_block<kThreads>(keys, n, kk, out, sel, st);
    fence_proxy_async_smem();
    __syncthreads();
    return total;
  };
  // One task's selection: the compute warps wait for the row's scores (`src`, n_src entries) and
  // rank them; the issue warp meanwhile runs `side` (its own waits are bounded).  Returns the count
  // (all threads), or -2 after a timeout.
  auto select_task = [&](int row, const float* src, int n_src, int kk, int cntP, int32_t* out,
                         auto&& side) -> int {
    if (warp == kW) {
      side();
    } else {
      if (tid == 0) wait_count(W.done + row, static_cast<unsigned>(n), abort_flag, kv.status);
      DSA_STAMP(6);  // task: the row's scores are complete
      int total = -1;
      if (!named_barrier_or(1, kCT, *abort_flag)) {
        load_keys(src, n_src);
        named_barrier(1, kCT);
        DSA_STAMP(7);  // task: keys loaded
        total = select_fast(kk, cntP, out);
      }
      if (tid == 0) s_red[3] = total;
    }
    __syncthreads();
    DSA_STAMP(8);  // task: ranked
    if (*abort_flag) return -2;
    const int total = s_red[3];
    return total >= 0 ? total : select_all(kk, out);
  };
  // A_t for a merge task (compute warps).  The workers appended every page of the row scoring at or
  // above its hint to the row's candidate list; when at least kk pages did, the row's kk best are
  // among them, so only the list is ranked: the kk best are marked in a bitmap and read out in
  // ascending order.  For the next step's hint the keys of rank C / 2 and C - 1 go to s_kmid and
  // s_klow, and the key of rank 1.5 kk - 1 to s_hint (0 when the list is shorter).  Otherwise (no hint yet, the scores moved below it, or more than
  // kCandCap candidates) returns -1 with the row's keys in place for the caller's full selection.
  // -2 after a timeout.  Bitmaps (rows of at most kBitsMax pages): ts.bits[0, w) A_t,
  // ts.bits[kBitsMax / 32, +w) P_t, the latter marked while the workers still score the row.
  auto select_merge = [&](int row, int kk, int cntP, int32_t* out, bool prepared) -> int {
    const int nwords = (n + 31) >> 5;
    uint32_t* abits = ts.bits;
    unsigned long long* cv = reinterpret_cast<unsigned long long*>(ts.hist);
    if (!prepared) merge_prep(row, cntP);
    if (tid == 0) wait_count(W.done + row, static_cast<unsigned>(n), abort_flag, kv.status);
    DSA_STAMP(6);  // task: the row's scores are complete
    if (named_barrier_or(1, kCT, *abort_flag)) return -2;
    // the workers whose shares meet the row: half a warp per worker's line (lane s reads slot s),
    // every round's load in flight; a warp claims the slots of all its workers' candidates at once
    constexpr int kRounds = (kMaxWorkers + 2 * kW - 1) / (2 * kW);
    int C = 0;
    // (fewer slots than workers leave some shares empty, their lines unwritten: no list then)
    bool over = workers > kMaxWorkers || T < workers;
    if (!over) {
      const int half = lane >> 4, sl = lane & 15;
      const int wlo = s_wlo, whi = s_whi;
      unsigned long long v[kRounds];
#pragma unroll
      for (int rr = 0; rr < kRounds; ++rr) {
        const int w = (rr * kW + warp) * 2 + half;
        const bool mine = w >= wlo && w <= whi;
        const size_t line = static_cast<size_t>(row) * kMaxWorkers + min(w, kMaxWorkers - 1);
        const unsigned long long x = __ldcg(W.cand + line * kWorkerSlots + sl);
        v[rr] = mine ? x : 0ull;
      }
      int wsum = 0;  // this warp's candidates before each round, then in all
      bool ovf = false;
      int off[kRounds];
#pragma unroll
      for (int rr = 0; rr < kRounds; ++rr) {
        const unsigned bal = __ballot_sync(0xffffffffu, v[rr] != 0ull && sl < kWorkerCand);
        ovf |= sl == kWorkerCand && v[rr] != 0ull;
        const int c_lo = __popc(bal & 0x7fffu), c_hi = __popc((bal >> 16) & 0x7fffu);
        off[rr] = wsum + (half ? c_lo : 0);
        wsum += c_lo + c_hi;
      }
      if (__any_sync(0xffffffffu, ovf) && lane == 0) s_hint = 1u;  // (an overflow, until below)
      int base = 0;
      if (lane == 0 && wsum > 0) base = atomicAdd(&ts.n_cand, wsum);
      base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
      for (int rr = 0; rr < kRounds; ++rr) {
        const int at = base + off[rr] + sl;
        if (sl < kWorkerCand && v[rr] != 0ull && at < kTopkMaxCand) cv[at] = v[rr];
      }
      named_barrier(1, kCT);
      C = ts.n_cand;
      over = s_hint != 0u || C > kTopkMaxCand;
    }
    if (over || C < kk || n > kBitsMax || kk < 1) {
      named_barrier(1, kCT);
      if (tid == 0) s_hint = 0u;
      load_keys(a.scores + static_cast<size_t>(row) * n, n);
      named_barrier(1, kCT);
      return -1;
    }
    if (tid == 0) {
      s_red[2] = C;
      s_kmid = s_klow = 0u;
      cv[C] = 0ull;  // the pair loads read one past an odd count
    }
    DSA_STAMP(7);  // task: candidates loaded
    named_barrier(1, kCT);
    // candidate i is among the kk best when fewer than kk rank values exceed its own; two threads
    // per candidate split the comparisons when the candidates are few
    const int tpc = C <= kCT / 2 ? 2 : 1;
    const int hint_rank = kk + kk / 2 - 1;
    for (int i0 = 0; i0 < C; i0 += kCT / tpc) {
      const int i = i0 + tid / tpc, part = tid % tpc;
      int r = 0;
      unsigned long long vi = 0ull;
      if (i < C) {
        vi = cv[i];
        const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(cv);
#pragma unroll 4
        for (int q2 = part; q2 < ((C + 1) >> 1); q2 += tpc) {
          const ulonglong2 x = c2[q2];
          r += (x.x > vi) + (x.y > vi);
        }
      }
      if (tpc == 2) r += __shfl_xor_sync(0xffffffffu, r, 1);
      if (i < C && part == 0) {
        if (r < kk) {
          const int pos = rank_pos_of(vi);
          atomicOr(&abits[pos >> 5], 1u << (pos & 31));
        }
        if (r == hint_rank) s_hint = static_cast<uint32_t>(vi >> 32);
        if (r == C / 2) s_kmid = static_cast<uint32_t>(vi >> 32);
        if (r == C - 1) s_klow = static_cast<uint32_t>(vi >> 32);
      }
    }
    named_barrier(1, kCT);
    // the marked positions in ascending order: thread t reads A's bitmap words [t*wpt, (t+1)*wpt)
    {
      const int wpt = (nwords + kCT - 1) / kCT;
      const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
      int cnt = 0;
      for (int w = w0; w < w1; ++w) cnt += __popc(abits[w]);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) ts.wcnt[warp] = incl;
      named_barrier(1, kCT);
      int at = incl - cnt;
      for (int w = 0; w < warp; ++w) at += ts.wcnt[w];
      for (int w = w0; w < w1; ++w)
        for (uint32_t m = abits[w]; m != 0u; m &= m - 1u) out[at++] = (w << 5) + __ffs(m) - 1;
    }
    DSA_STAMP(14);  // task: A_t ranked (compute warps)
    return kk;      // exactly kk candidates rank below kk (C >= kk, rank values distinct)
  };
  auto load_plist = [&](int row) -> int {
    const int cntP = min(max(a.spec_count[row], 0), kp);
    for (int i = tid; i < cntP; i += kThreads) pl[i] = a.spec_idx[static_cast<size_t>(row) * kp + i];
    return cntP;
  };

  // The counters go back to zero once every CTA has arrived at the exit count: the last to
  // arrive resets them.  A CTA arrives after its last wait on a counter; every increment of the
  // counters has then been seen by a wait of some CTA that arrived before it, so none is in flight.
  auto reset_counters = [&]() {
    for (int r = 0; r < rows; ++r) {
      W.done[r] = 0u;
      W.sdone[r] = 0u;
    }
    *W.exit = 0u;
  };
  bool arrived = false;  // (uniform) the CTA has arrived at the exit count
  for (int task = split ? (cta < n_tasks ? cta : n_tasks) : cta; task < n_tasks;
       task += split ? n_tasks : grid) {
    __syncthreads();  // the previous task's shared data are no longer read
    if (task >= rows * G) {
      // ---- P_{t+1} = top-k_pred of the new predictions
      const int row = task - rows * G;
      const int cntP = load_plist(row);
      __syncthreads();
      const int total = select_task(row, W.pred + static_cast<size_t>(row) * kv.max_pages,
                                    min(n, kv.max_pages), kp, cntP,
                                    a.next_idx + static_cast<size_t>(row) * kp, [] {});
      if (total == -2) break;
      if (tid == 0) a.next_count[row] = total;
      continue;
    }
    // ---- (row, query head): A_t, the missed pages, the merge
    const int row = task / G, g = task - row * G;
    const int b = row / kv.Hkv;
    const int L = request_len(kv, b);
    const int npos = (L + page - 1) / page;
    const size_t qhead = static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(row % kv.Hkv) * G + g;
    const bool prepared = pre && task == cta;  // its first steps taken in the worker phase
    const int cntP = prepared ? s_cntp : load_plist(row);
    if (!prepared) __syncthreads();
    DSA_STAMP(5);  // task (merge): start
    const float* recs = a.partials + static_cast<size_t>(row) * kp * G * kRecordFloats;
    // the issue warp: once the row's records are written, query head g's of them on chip
    auto fetch_records = [&]() {
      if (!a.rec_smem) return;
      if (lane == 0) wait_count(W.sdone + row, static_cast<unsigned>(cntP), abort_flag, kv.status);
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) return;
      constexpr int kPieces = kRecordFloats / 4;
      const uint32_t dst = smem_u32(srec);
      for (int e = lane; e < cntP * kPieces; e += 32) {
        const int i = e / kPieces, c = e - i * kPieces;
        cp_async16(dst + static_cast<uint32_t>(i * kRecordFloats + c * 4) * 4u,
                   recs + (static_cast<size_t>(i) * G + g) * kRecordFloats + c * 4);
      }
      cp_async_wait_all();
    };
    int cntA;
    if (warp == kW) {
      fetch_records();
    } else {
      const int got = select_merge(row, a.k, cntP, sA, prepared);
      if (tid == 0) s_red[3] = got;
    }
    __syncthreads();
    if (*abort_flag) break;
    DSA_STAMP(8);  // task: ranked
    // with the records on chip the waits on the row's counters are behind this CTA: in its last
    // task the issue warp arrives at the exit count now and reads the ticket once it has issued
    // the missed pages, which takes the arrival off the launch's tail
    const bool early_exit = a.rec_smem && task + (split ? n_tasks : grid) >= n_tasks;
    unsigned exit_ticket = 0u;
    if (early_exit && warp == kW && lane == 0) exit_ticket = atomicAdd(W.exit, 1u);
    arrived = early_exit;
    cntA = s_red[3];
    const bool bits_ok = cntA >= 0;  // the A_t and P_t bitmaps hold
    if (cntA == -1) {  // the keys are in place: P_t's bound over them, else every key
      DSA_STAMP(15);   // task: A_t from the keys
      if (warp < kW) {
        const int t = select_fast(a.k, cntP, sA);
        if (tid == 0) s_red[3] = t;
      }
      __syncthreads();
      cntA = s_red[3];
      if (cntA < 0) cntA = select_all(a.k, sA);
    }
    if (g == 0) {  // the first query head's task publishes A_t
      for (int i = tid; i < a.k; i += kThreads) a.idx[static_cast<size_t>(row) * a.k + i] = sA[i];
      if (tid == 0) a.count[row] = cntA;
    }
    if (g == 0) {  // the next step's hint (any value is safe; it only decides the speed)
      if (!bits_ok) {  // from the row's k best (the keys are still in place): ranks k / 2, k - 1
        uint32_t* kA = reinterpret_cast<uint32_t*>(mlist);  // their keys, staged once
        if (tid == 0) s_kmid = s_klow = 0u;
        for (int i = tid; i < cntA; i += kThreads) kA[i] = keys[sA[i]];
        __syncthreads();
        for (int i0 = 0; i0 < cntA; i0 += kThreads / 4) {  // four threads per key
          const int i = i0 + (tid >> 2), part = tid & 3;
          int r = 0;
          if (i < cntA) {
            const uint32_t ki = kA[i];
            for (int j = part; j < cntA; j += 4) r += kA[j] > ki || (kA[j] == ki && j < i);
          }
          r += __shfl_xor_sync(0xffffffffu, r, 1);
          r += __shfl_xor_sync(0xffffffffu, r, 2);
          if (i < cntA && part == 0) {
            if (r == cntA / 2) s_kmid = kA[i];
            if (r == cntA - 1) s_klow = kA[i];
          }
        }
        __syncthreads();
      }
      if (tid == 0) {
        // the exact key of rank 1.5k - 1 when the list reached it.  Else, taking the top scores'
        // log-rank as linear in the score (a drop of d per doubling of the rank, d measured from
        // rank seen / 2 to seen - 1), the score where rank 1.75k would stand
        const int seen = bits_ok ? s_red[2] : cntA;
        uint32_t h = s_hint;
        if (h == 0u && seen >= 4 && s_kmid != 0u && s_klow != 0u) {
          const float mid = key_score(s_kmid), low = key_score(s_klow);
          const float doublings = log2f(static_cast<float>(seen) / (seen / 2 + 1));
          const float d = (mid - low) / doublings;
          const float want = low - d * log2f(1.75f * a.k / static_cast<float>(seen));
          h = (isfinite(want) && want < low) ? score_key(want) : s_klow;
        }
        W.hint[row] = h;
      }
    }
    cntA = min(max(cntA, 0), a.k);
    // merged speculative parts (warp 0): P slots whose page is in A (every slot in superset
    // mode); missed pages (warp 1): A \ P (both lists are ascending)
    if (warp == 0) {
      int np = 0;
      for (int base = 0; base < cntP; base += 32) {
        const int i = base + lane;
        const bool take =
            i < cntP && (a.superset ||
                         (bits_ok ? pl[i] >= 0 && pl[i] < n &&
                                        ((ts.bits[pl[i] >> 5] >> (pl[i] & 31)) & 1u) != 0u
                                  : contains_sorted(sA, cntA, pl[i])));
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        if (take) parts[np + __popc(bal & below)] = i;
        np += __popc(bal);
      }
      if (lane == 0) s_red[0] = np;
    } else if (warp == 1) {
      int nm = 0;
      for (int base = 0; base < cntA; base += 32) {
        const int i = base + lane;
        const bool miss =
            i < cntA && !(bits_ok ? ((ts.bits[kBitsMax / 32 + (sA[i] >> 5)] >> (sA[i] & 31)) & 1u) != 0u
                                  : contains_sorted(pl, cntP, sA[i]));
        const unsigned bal = __ballot_sync(0xffffffffu, miss);
        if (miss) mlist[nm + __popc(bal & below)] = sA[i];
        nm += __popc(bal);
      }
      if (lane == 0) s_red[1] = nm;
    }
    __syncthreads();
    DSA_STAMP(9);  // task: merged and missed lists
    const int n_parts = s_red[0], n_miss = s_red[1];
    // ---- the missed pages through the ring: warp w < S attends pages w, w + S, ... into one
    // state and leaves query head g's part of it (unnormalised O, max in log2 units, sum) in
    // wst[w]
    if (warp == kW) {
      if (lane == 0) {
        for (int i = 0; i < n_miss; ++i)
          if (!issue(ring + i, row, mlist[i], true, npos)) break;
        if (early_exit && exit_ticket == gridDim.x - 1) reset_counters();
      }
      __syncwarp();
    } else {
      float* ws = wst + warp * kWs;
      if (lane == 0) ws[1] = 0.f;
      if (warp < S && warp < n_miss) {
        uint32_t qa[8][4];
        warp_q(row, qa);
        WarpSoftmaxState st;
        state_init(st);
        bool ok = true;
        for (int i = warp; i < n_miss && ok; i += S) ok = attend_item(ring + i, L, qa, st) != -2;
        state_finish(st);
        // row g is row g % 8 of the lanes' first (g < 8) or second half; the halves are chosen
        // with constant indices, so the state stays in registers
        if ((lane >> 2) == (g & 7)) {
          const int c0 = (lane & 3) * 2;
          const bool hi = g >= 8;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            *reinterpret_cast<float2*>(ws + 4 + jj * 8 + c0) =
                hi ? make_float2(st.o[jj][2], st.o[jj][3]) : make_float2(st.o[jj][0], st.o[jj][1]);
          if ((lane & 3) == 0) {
            ws[0] = hi ? st.m[1] : st.m[0];
            ws[1] = hi ? st.l[1] : st.l[0];
          }
        }
      }
    }
    ring += n_miss;
    __syncthreads();
    DSA_STAMP(10);  // task: missed pages attended
    if (*abort_flag) break;
    // without the on-chip copy, the records are read from L2 once the row's are complete
    if (!a.rec_smem) {
      if (tid == 0) wait_count(W.sdone + row, static_cast<unsigned>(cntP), abort_flag, kv.status);
      __syncthreads();
      if (*abort_flag) break;
    }

    DSA_STAMP(11);  // task: records ready
    float wm = -INFINITY, wl = 0.f;  // this warp's state: max (log2 units), sum, unnormalised O
    float4 wo = make_float4(0.f, 0.f, 0.f, 0.f);
    auto absorb = [&](float m2, float l, float4 o) {  // adds a part (max m2, sum l, O = o * l)
      if (!(l > 0.f)) return;
      const float mn = fmaxf(wm, m2);
      const float f_old = wm == -INFINITY ? 0.f : fast_exp2(wm - mn);
      const float f_new = fast_exp2(m2 - mn) * l;
      wl = wl * f_old + f_new;
      wo.x = wo.x * f_old + o.x * f_new;
      wo.y = wo.y * f_old + o.y * f_new;
      wo.z = wo.z * f_old + o.z * f_new;
      wo.w = wo.w * f_old + o.w * f_new;
      wm = mn;
    };
    // adds a sum of parts: max m2, sum l, unnormalised O o (both relative to m2)
    auto absorb_sum = [&](float m2, float l, float4 o) {
      const float mn = fmaxf(wm, m2);
      const float f_old = wm == -INFINITY ? 0.f : fast_exp2(wm - mn);
      const float f = fast_exp2(m2 - mn);
      wl = wl * f_old + l * f;
      wo.x = wo.x * f_old + o.x * f;
      wo.y = wo.y * f_old + o.y * f;
      wo.z = wo.z * f_old + o.z * f;
      wo.w = wo.w * f_old + o.w * f;
      wm = mn;
    };
    float* ws = wst + warp * kWs;
    if (warp < kW && ws[1] > 0.f) {  // this warp's missed pages
      const float inv = 1.f / ws[1];
      const float4 o = *(reinterpret_cast<const float4*>(ws + 4) + lane);
      absorb(ws[0], ws[1], make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv));
    }
    // ---- speculative records, kRoundRecs per warp round: each record's weight against the
    // round's largest max (independent exponentials), then one merge into the warp's state
    for (int i0 = warp; i0 < n_parts; i0 += kRoundRecs * kWarps) {
      float2 ml[kRoundRecs];
      float4 ov[kRoundRecs];
#pragma unroll
      for (int u = 0; u < kRoundRecs; ++u) {
        const int i = i0 + u * kWarps;
        ml[u] = make_float2(-INFINITY, 0.f);
        ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n_parts) {
          if (a.rec_smem) {
            const float* r = srec + parts[i] * kRecordFloats;
            ml[u] = *reinterpret_cast<const float2*>(r + 128);
            ov[u] = *(reinterpret_cast<const float4*>(r) + lane);
          } else {
            const float* r = recs + (static_cast<size_t>(parts[i]) * G + g) * kRecordFloats;
            ml[u] = __ldcg(reinterpret_cast<const float2*>(r + 128));
            ov[u] = __ldcg(reinterpret_cast<const float4*>(r) + lane);
          }
        }
      }
      float mr = -INFINITY;  // (every lane holds the same m and l: the branches are uniform)
#pragma unroll
      for (int u = 0; u < kRoundRecs; ++u)
        if (ml[u].y > 0.f) mr = fmaxf(mr, ml[u].x * kLog2e);
      if (mr == -INFINITY) continue;
      float rl = 0.f;
      float4 ro = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < kRoundRecs; ++u) {
        const float f = ml[u].y > 0.f ? fast_exp2(ml[u].x * kLog2e - mr) * ml[u].y : 0.f;
        rl += f;
        ro.x += f * ov[u].x;
        ro.y += f * ov[u].y;
        ro.z += f * ov[u].z;
        ro.w += f * ov[u].w;
      }
      absorb_sum(mr, rl, ro);
    }
    DSA_STAMP(19);  // task: thread 0's warp has merged its records
    __syncwarp();
    if (lane == 0) {
      ws[0] = wm;
      ws[1] = wl;
    }
    *reinterpret_cast<float4*>(ws + 4 + lane * 4) = wo;
    __syncthreads();
    DSA_STAMP(20);  // task: every warp's state stored (barrier)
    // ---- combine the warps' states
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (wst[w * kWs + 1] > 0.f) M = fmaxf(M, wst[w * kWs]);
    if (tid < kHeadDim) {
      float o = 0.f, lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float lw = wst[w * kWs + 1];
        if (!(lw > 0.f)) continue;
        const float f = fast_exp2(wst[w * kWs] - M);
        lsum += lw * f;
        o += wst[w * kWs + 4 + tid] * f;
      }
      a.out[qhead * kHeadDim + tid] = lsum > 0.f ? o / lsum : 0.f;
      if (tid == 0) {
        a.m[qhead] = lsum > 0.f ? M * kLn2 : -INFINITY;
        a.l[qhead] = lsum;
      }
    }
    DSA_STAMP(12);  // task: output written
  }
  __syncthreads();
  if (*abort_flag) {
    drain();
    return;
  }

  // ---- the CTAs that have not arrived yet (workers, selections) arrive on their way out
  if (tid == 0 && !arrived) {
    __threadfence();
    if (atomicAdd(W.exit, 1u) == gridDim.x - 1) reset_counters();
  }
  DSA_STAMP(13);  // end
  DSA_TRACE_END(g_trace_prr);
}

// The deepest ring, with a task's records on chip if possible, that fits the shared-memory limit.
struct Shape {
  int stages;
  bool rec_smem;
};
Shape choose_shape(int page, int n, int k_pred, size_t static_bytes) {
  for (int pass = 0; pass < 2; ++pass)
    for (int S = kMaxStages; S >= 1; --S)
      if (slayout(page, n, k_pred, S, pass == 0).total + static_bytes <= kPrrSmemLimit)
        return Shape{S, pass == 0};
  return Shape{0, false};
}

size_t static_smem() {
  cudaFuncAttributes fa = {};
  return cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(prr_step_kernel)) == cudaSuccess
             ? fa.sharedSizeBytes
             : 24 * 1024;
}

}  // namespace

size_t prr_step_workspace_bytes(int rows, int max_pages) {
  return ws_layout(rows, max_pages).total;
}

size_t prr_step_counter_bytes(int rows) { return ws_layout(rows, 1).counters; }

size_t prr_step_smem_bytes(int page, int n, int k_pred) {
  const size_t stat = static_smem();
  const Shape sh = choose_shape(page, n, k_pred, stat);
  return sh.stages > 0 ? slayout(page, n, k_pred, sh.stages, sh.rec_smem).total + stat : SIZE_MAX;
}

cudaError_t launch_prr_step(const CUtensorMap& tmK, const CUtensorMap& tmV, const PrrStepArgs& s,
                            void* workspace, cudaStream_t stream) {
  PrrArgs a;
  a.kv = s.kv;
  a.q = s.q;
  a.meta = s.meta;
  a.scores = s.scores;
  a.stride = s.stride;
  a.ell = s.ell;
  a.trend = s.trend;
  a.alpha = s.alpha;
  a.beta = s.beta;
  a.gamma = s.gamma;
  a.pred = s.pred;
  a.spec_idx = s.spec_idx;
  a.spec_count = s.spec_count;
  a.k_pred = s.k_pred;
  a.partials = s.partials;
  a.idx = s.idx;
  a.count = s.count;
  a.k = s.k;
  a.next_idx = s.next_idx;
  a.next_count = s.next_count;
  a.superset = s.superset;
  a.scale_log2 = s.scale_log2;
  a.out = s.out;
  a.m = s.m;
  a.l = s.l;
  const WsLayout wl = ws_layout(s.kv.B * s.kv.Hkv, s.kv.max_pages);
  char* w = static_cast<char*>(workspace);
  a.ws.exit = reinterpret_cast<unsigned*>(w + wl.exit_off);
  a.ws.done = reinterpret_cast<unsigned*>(w + wl.done_off);
  a.ws.sdone = reinterpret_cast<unsigned*>(w + wl.sdone_off);
  a.ws.hint = reinterpret_cast<uint32_t*>(w + wl.hint_off);
  a.ws.cand = reinterpret_cast<unsigned long long*>(w + wl.cand_off);
  a.ws.pred = reinterpret_cast<float*>(w + wl.pred_off);
  const Shape sh = choose_shape(s.kv.p, s.stride, s.k_pred, static_smem());
  if (sh.stages < 1) return cudaErrorInvalidConfiguration;
  a.stages = sh.stages;
  a.rec_smem = sh.rec_smem ? 1 : 0;
  const size_t bytes = slayout(s.kv.p, s.stride, s.k_pred, a.stages, sh.rec_smem).total;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(prr_step_kernel), bytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prr_step_kernel, kThreads,
                                                         bytes)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // CTAs wait on per-row counters that other CTAs advance, so every CTA must be resident at once:
  // the grid is one CTA per SM and at least one fits on each.  The launch is a programmatic one
  // without the cooperative attribute (with it, the launch overlapped nothing): its CTAs take SMs
  // as the previous kernel of the stream leaves them, only after every CTA of that kernel has
  // started, and wait for it to finish at grid_dependency_wait; once it has, every SM is free for
  // the rest of this grid.  The counter
  // waits are bounded (DSA_STATUS_TIMEOUT) should another stream hold SMs for longer.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  // programmatic stream serialization: the launch may begin while the previous kernel of the
  // stream runs; the kernel waits for it (grid_dependency_wait) before its first global read
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prr_step_kernel, tmK, tmV, a);
}

}  // namespace dsa

#ifdef DSA_TIMELINE
// Phase-trace accessors of the traced library (see DSA_TRACE_BEGIN).
extern "C" int dsa_trace_read_prr(void* host, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(
      host, dsa::g_trace_prr, bytes < sizeof(dsa::g_trace_prr) ? bytes : sizeof(dsa::g_trace_prr)));
}
extern "C" int dsa_trace_clear_prr() {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, dsa::g_trace_prr);
  return static_cast<int>(e == cudaSuccess ? cudaMemset(p, 0, sizeof(dsa::g_trace_prr)) : e);
}
#endif
