// One whole PRR decode step (t >= 1) in a single cooperative launch ("Predict, Reuse, and Repair"
// §3: speculation over the predicted set, predictor update, repair and merge).
//
// Every CTA (one per SM, all resident) runs three phases separated by two grid barriers:
//   1. its share of the speculative per-page attention over P_t (one TMA-staged page per item,
//      the whole query group as the m16 tile) while it scores its equal share of the (row, page)
//      metadata records with the scoring kernel's exact arithmetic;
//   2. per row, one CTA selects A_t = top-k of the scores and another updates the EMA predictor
//      and selects P_{t+1} = top-k_pred of the prediction (the selection kernels' code);
//   3. per (row, query head), one CTA attends to the missed pages A_t \ P_t on the CUDA cores and
//      merges that part with the speculative records of A_t ∩ P_t (or all of P_t) by log-sum-exp.
// Barrier waits are bounded: a CTA that gives up raises DSA_STATUS_TIMEOUT and skips the rest.
// The barrier counters live in the caller's workspace; the last CTA out resets them to zero.
#include "attn_core.cuh"
#include "internal.h"
#include "score_core.cuh"
#include "select.cuh"

namespace dsa {
namespace {

constexpr int kPW = 8;                     // compute warps of phase 1
constexpr int kPThreads = (kPW + 1) * 32;  // + one TMA issue warp; phases 2 and 3 use all nine
constexpr int kPWarps = kPThreads / 32;
constexpr int kPStages = 2;
constexpr int kPGroups = kPW * 32 / 8;  // scoring record groups of 8 lanes
constexpr int kCandCap = kTopkMaxCand;  // candidates kept per row for the selection of A_t
constexpr int kScoutEvery = 19;  // every 19th CTA (8 of 152) is a scout that does not score
constexpr int kScoreRecs = 128;  // metadata records a CTA's scoring stages in shared memory at once
constexpr int kEmaCap = 1024;  // EMA updates a CTA stages on chip during scoring (its slot share)

struct PLayout {
  // phase 1
  uint32_t stage_off, merge_off, q_off, qbar_off, wt_off, sps_off, ppk_off, bar_off, ctl_off;
  // phase 3
  uint32_t sp_off, sa_off, list_off, part_off, qh_off, ws_off, bmp_off, bma_off, rec_off, keys_off;
  // the EMA updates staged from phase 1 to the end of phase 2: past every other region
  uint32_t ema_off, total;
};

__host__ __device__ inline uint32_t up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline PLayout playout(int page, int G, int n, int k, int k_pred) {
  PLayout L;
  L.stage_off = 0;
  L.merge_off = up(kPStages * 512u * page, 1024);
  uint32_t merge_bytes = kPW * G * (kHeadDim + 2) * 4u;
  if (merge_bytes < kScoreRecs * 512u) merge_bytes = kScoreRecs * 512u;  // scoring record buffer
  L.q_off = up(L.merge_off + merge_bytes, 16);
  L.qbar_off = up(L.q_off + 16u * kQStride * 2u, 16);
  L.wt_off = up(L.qbar_off + kHeadDim * 4u, 16);
  L.sps_off = up(L.wt_off + (kPW + 1) * 16 * 4u, 16);
  L.ppk_off = up(L.sps_off + 4u * k_pred, 16);
  L.bar_off = up(L.ppk_off + 4u * k_pred, 16);
  L.ctl_off = L.bar_off + 2 * kPStages * 8u;
  const uint32_t p1_end = L.ctl_off + 2 * kPStages * 4u;
  // phase 3
  L.sp_off = 0;
  L.sa_off = up(4u * k_pred, 16);
  L.list_off = up(L.sa_off + 4u * k, 16);
  L.part_off = up(L.list_off + 8u * k, 16);
  L.qh_off = up(L.part_off + 4u * k_pred, 16);
  L.ws_off = up(L.qh_off + 4u * kHeadDim, 16);
  L.bmp_off = up(L.ws_off + kPWarps * (kHeadDim + 4) * 4u, 16);
  L.bma_off = up(L.bmp_off + 4u * ((n + 31) / 32), 16);
  L.rec_off = up(L.bma_off + 4u * ((n + 31) / 32), 16);
  // keys [n] of a full-row selection share the record area: a task that needs one selects before
  // it fetches the records
  L.keys_off = L.rec_off;
  uint32_t rec_bytes = 4u * kRecordFloats * k_pred;
  if (rec_bytes < 4u * static_cast<uint32_t>(n)) rec_bytes = 4u * static_cast<uint32_t>(n);
  const uint32_t p3_end = L.rec_off + rec_bytes;
  uint32_t t = p1_end;
  if (p3_end > t) t = p3_end;
  L.ema_off = up(t, 16);
  L.total = L.ema_off + 3u * 4u * kEmaCap + 1024u;  // + alignment slack
  return L;
}

DSA_DEV unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Arrival on a monotonically counting word, after every write of this CTA so far.
DSA_DEV void grid_arrive(unsigned* ctr, volatile int* abort) {
  __syncthreads();
  if (threadIdx.x == 0 && !*abort) {
    __threadfence();  // this CTA's writes (ordered before by the CTA barrier) become visible
    atomicAdd(ctr, 1u);
  }
}

// Waits until the word reaches `target` (compared as a sequence number, so a word that wrapped
// around still orders).  Bounded: gives up after kWaitLimitNs, raising DSA_STATUS_TIMEOUT.
// Returns false when this CTA (or an earlier wait of it) gave up.
DSA_DEV bool grid_wait(unsigned* ctr, unsigned target, volatile int* abort, int32_t* status) {
  if (threadIdx.x == 0 && !*abort) {
    const unsigned long long t0 = global_timer_ns();
    while (static_cast<int>(ld_acquire(ctr) - target) < 0) {
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        raise_status(status, DSA_STATUS_TIMEOUT);
        break;
      }
      __nanosleep(100);
    }
  }
  __syncthreads();
  return !*abort;
}

// Grid-wide barrier: arrive, then wait until every CTA has.
DSA_DEV bool grid_barrier(unsigned* ctr, unsigned target, volatile int* abort, int32_t* status) {
  grid_arrive(ctr, abort);
  return grid_wait(ctr, target, abort, status);
}

struct PrrArgs {
  KvView kv;
  const __nv_bfloat16* kpool;  // bf16 [P][Hkv][p][128]
  const __nv_bfloat16* vpool;
  const __nv_bfloat16* q;
  const uint8_t* meta;
  float* scores;
  int stride;  // score / EMA row stride = candidates per row
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
  unsigned* sync;        // [0] barrier 1, [1] barrier 2, [2] exit count
  unsigned* cand_cnt;    // [rows] candidates for A_t appended (zero on entry, left zero)
  uint2* cand;           // [rows][kCandCap] (key, index)
  unsigned* cand_cnt2;   // [rows] candidates for P_{t+1} (zero on entry, left zero)
  uint2* cand2;          // [rows][kCandCap]
};

__global__ void __launch_bounds__(kPThreads, 1)
    prr_step_kernel(const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const PrrArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023u) & ~static_cast<uintptr_t>(1023u));
  __shared__ SelectAnyScratch<kPThreads> sel_scratch;
  __shared__ int s_abort, s_issued, s_red[33];
  __shared__ unsigned s_t0key, s_t1key;
  __shared__ unsigned s_cand[4];  // scoring's candidate counts of a round: CTA-local, CTA base
  __shared__ float s_f[kPWarps];
  const KvView& kv = a.kv;
  const int page = kv.p, G = kv.G, tiles = page / 16;
  const int rows = kv.B * kv.Hkv;
  const int n = a.stride;
  const PLayout lay = playout(page, G, n, a.k, a.k_pred);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t stage_bytes = 512u * page;

  // ================================================================ phase 1
  float* sO = reinterpret_cast<float*>(smem + lay.merge_off);  // [kPW][G][128]
  float* sM = sO + kPW * G * kHeadDim;                          // [kPW][G]
  float* sL = sM + kPW * G;                                     // [kPW][G]
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + lay.q_off);
  float* qbar = reinterpret_cast<float*>(smem + lay.qbar_off);
  float* wt = reinterpret_cast<float*>(smem + lay.wt_off);  // [kPW][16] warp weight / l
  uint32_t* spk = reinterpret_cast<uint32_t*>(smem + lay.sps_off);  // keys of P_t's true scores
  uint32_t* ppk = reinterpret_cast<uint32_t*>(smem + lay.ppk_off);  // ... of their predictions
  float* st_ell = reinterpret_cast<float*>(smem + lay.ema_off);     // staged EMA updates [kEmaCap]
  float* st_v = st_ell + kEmaCap;
  float* st_pred = st_v + kEmaCap;
  // This CTA's equal share [s_beg, s_end) of the (row, page) slots, for scoring and the EMA.  On
  // a full grid every kScoutEvery-th CTA is a scout that takes no share: it goes straight to its
  // speculative pages, so the code of that part is in L2 before the scoring CTAs reach it.
  const long long T = static_cast<long long>(rows) * n;
  const int grid = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const bool scouts = grid >= 2 * kScoutEvery;
  const bool scout = scouts && cta % kScoutEvery == 0;
  const int scorers = scouts ? grid - (grid + kScoutEvery - 1) / kScoutEvery : grid;
  const int rank = scouts ? cta - (cta / kScoutEvery + 1) : cta;  // among the scorers
  const long long s_beg = scout ? 0 : static_cast<long long>(rank) * T / scorers;
  const long long s_end = scout ? 0 : static_cast<long long>(rank + 1) * T / scorers;
  // the EMA update rides along with scoring when every share fits on chip and enough CTAs take the
  // roles of phase 2; its writes wait for the second barrier (until then the old state is read)
  const bool roles = grid > 2 * rows;
  const bool ema1 = roles && (T + scorers - 1) / scorers <= kEmaCap;
  // Roles after the first barrier (with more than 2 rows CTAs): CTA rows + r selects P_{t+1} of
  // row r; every other CTA repairs (row, query head) tasks, selecting A_t of the task's row itself
  // from the candidate list, so the repair waits for no further barrier.
  const bool p_role = roles && cta >= rows && cta < 2 * rows;
  const int rep_first = !roles ? cta : p_role ? -1 : (cta < rows ? cta : cta - rows);
  const int rep_step = roles ? grid - rows : grid;
  // A scout without a repair task of its own rehearses one (its writes suppressed) between its
  // arrival at the first barrier and the end: the repair code is then in L2 when the repair CTAs
  // reach it after the barrier.  It needs nothing behind the barrier.  The odd-numbered ones past
  // every repair task (CTA >= rows (G + 1)) attend no speculative pages either and rehearse from
  // the start; the speculative items go round-robin over the other CTAs.
  const bool rehearse =
      roles && scout && !p_role && !(rep_first >= 0 && rep_first < rows * G) && rows * G > 0;
  const bool dry = rehearse;
  auto early_rehearser = [&](int c) {
    return roles && scouts && c % kScoutEvery == 0 && (c / kScoutEvery) % 2 == 1 &&
           c >= rows * (G + 1);
  };
  int n_early = 0, early_before = 0;
  for (int c = kScoutEvery; c < grid; c += 2 * kScoutEvery)
    if (early_rehearser(c)) {
      ++n_early;
      if (c < cta) ++early_before;
    }
  const bool early = early_rehearser(cta);
  const int item_ctas = grid - n_early;
  // rank among the CTAs with speculative items: the scouts first, so that the ones left with an
  // extra item (the first items % item_ctas) are CTAs that do not score
  const int n_scouts = scouts ? (grid + kScoutEvery - 1) / kScoutEvery : 0;
  const int irank = !scouts ? cta
                    : scout ? cta / kScoutEvery - early_before
                            : n_scouts - n_early + rank;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bar_off);  // [S] full, [S] empty
  volatile int* stage_ok = reinterpret_cast<int*>(smem + lay.ctl_off);  // [S]: -1 none, 0, 1
  volatile int* stage_pos = stage_ok + kPStages;
  if (warp == 1 && lane < 8) {
    // phase 1 reads these first: start their address translations at once
    const long long sb = s_beg;
    const int row = static_cast<int>(sb / n);
    const int b = row / kv.Hkv;
    const void* p = nullptr;
    switch (lane) {
      case 0: p = a.spec_count + row; break;
      case 1: p = a.spec_idx + static_cast<size_t>(row) * a.k_pred; break;
      case 2: p = kv.page_table + static_cast<size_t>(b) * kv.max_pages; break;
      case 3: p = kv.seq_lens + b; break;
      case 4: p = a.scores + sb; break;
      case 5: p = a.ell + sb; break;
      case 6: p = a.trend + sb; break;
      default: p = a.q + static_cast<size_t>(b) * kv.Hq * kHeadDim; break;
    }
    prefetch_l2(p);
  }
  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[kPStages + s]), kPW);
    }
    fence_mbar_init();
    s_abort = 0;
    s_cand[0] = 0u;
    s_cand[1] = 0u;
    s_issued = 0;
  }
  __syncthreads();
  const int n_items_total = rows * a.k_pred;
  const int my_items =
      !early && irank < n_items_total ? (n_items_total - 1 - irank) / item_ctas + 1 : 0;

  if (warp == kPW) {
    // ---- TMA issue warp: the speculative pages of this CTA's items
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      for (int j = 0; j < my_items; ++j) {
        const int it = irank + j * item_ctas;
        const int row = it / a.k_pred, slot = it - row * a.k_pred;
        const int b = row / kv.Hkv, h = row % kv.Hkv;
        const int s = j % kPStages, u = j / kPStages;
        if (u > 0 && !mbar_wait(smem_u32(&bars[kPStages + s]), (u - 1) & 1, abort_flag, kv.status))
          break;
        const int cnt = min(max(a.spec_count[row], 0), a.k_pred);
        int okv = -1, pos = -1, phys = 0;
        if (slot < cnt) {
          pos = a.spec_idx[static_cast<size_t>(row) * a.k_pred + slot];
          const int npos = (request_len(kv, b) + page - 1) / page;
          okv = lookup_page(kv, b, pos, npos, &phys) ? 1 : 0;
        }
        const uint32_t full = smem_u32(&bars[s]);
        stage_ok[s] = okv;
        stage_pos[s] = pos;
        if (okv == 1) {
          const uint32_t dst = smem_base + s * stage_bytes;
          const int row0 = (phys * kv.Hkv + h) * page;
          mbar_arrive_expect_tx(full, stage_bytes);
          tma_load_page(dst, &tmK, row0, full);
          tma_load_page(dst + 2 * page * 128, &tmV, row0, full);
        } else {
          mbar_arrive(full);
        }
        *reinterpret_cast<volatile int*>(&s_issued) = j + 1;
      }
    }
    __syncwarp();
  } else {
    // copies the query rows of speculative item j to shared memory, one 16-byte piece per thread
    // (row tid / 16, dims 8 (tid % 16) ...; rows past the group are zero).  The first item's are
    // copied before scoring, so they are on chip when its page lands.
    auto stage_q = [&](int j) {
      const int row = (irank + j * item_ctas) / a.k_pred;
      const int b = row / kv.Hkv, h = row % kv.Hkv;
      const int r = tid >> 4, c = tid & 15;
      __nv_bfloat16* dst = sQ + r * kQStride + c * 8;
      if (r < G)
        cp_async16(smem_u32(dst),
                   a.q + (static_cast<size_t>(b) * kv.Hq + h * G + r) * kHeadDim + c * 8);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    };
    if (my_items > 0) stage_q(0);
    // ---- scoring: this CTA's equal share of the (row, page) slots.  Per segment (the part of
    // one row) the loads go out in three waves of independent requests: (1) the group query,
    // P_t's positions, the chunk's page-table entries and EMA state; (2) the chunk's metadata
    // records (copied asynchronously into the merge area, idle until the speculative attention)
    // and P_t's page-table entries; (3) P_t's metadata records and EMA state.  Record groups of
    // 8 lanes (32 per CTA): group gid takes P_t slots gid + 32 i and chunk slots j0 + gid + 32 i.
    // Each lane copies and later reads the same 64 bytes of a staged record: no barrier needed.
    const int gl = lane & 7, gid = tid >> 3;
    constexpr int kPB = 256 / kPGroups;  // P_t slots per group (k_pred <= 256)
    constexpr int kCB = kScoreRecs / kPGroups;  // chunk slots per group per wave
    constexpr int kPR = 4;  // P_t records in flight per group in wave 3 (divides kPB)
    const uint32_t rbuf = smem_u32(sO);
    // copies this lane's part of record `rec` into buffer slot `slot` / reads it back
    auto stage_record = [&](size_t rec, int slot) {
      const uint8_t* src = a.meta + rec * 512;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        cp_async16(rbuf + slot * 512 + (gl + 8 * c) * 16, src + (gl + 8 * c) * 16);
    };
    auto staged_record = [&](int slot, uint4 (&raw)[4]) {
      const uint4* p =
          reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(sO) + slot * 512);
#pragma unroll
      for (int c = 0; c < 4; ++c) raw[c] = p[gl + 8 * c];
    };
    auto score_share = [&]() {
      for (long long seg = s_beg; seg < s_end;) {
        const int row = static_cast<int>(seg / n);
        const int j0 = static_cast<int>(seg - static_cast<long long>(row) * n);
        const int j1 = static_cast<int>(min(s_end - static_cast<long long>(row) * n,
                                            static_cast<long long>(n)));
        seg = static_cast<long long>(row) * n + j1;
        const int b = row / kv.Hkv, h = row % kv.Hkv;
        const int nl = (request_len(kv, b) + page - 1) / page;
        const int32_t* table = kv.page_table + static_cast<size_t>(b) * kv.max_pages;
        float* outs = a.scores + static_cast<size_t>(row) * n;
        const int cntP = min(max(a.spec_count[row], 0), a.k_pred);
        const int32_t* P = a.spec_idx + static_cast<size_t>(row) * a.k_pred;
        const float* ell_r = a.ell + static_cast<size_t>(row) * n;
        const float* v_r = a.trend + static_cast<size_t>(row) * n;
        named_barrier(1, kPW * 32);  // qbar, spk and ppk of the previous segment are no longer read

        // ---- wave 1
        float qacc = 0.f;
        if (tid < kHeadDim) {
          const __nv_bfloat16* qg = a.q + (static_cast<size_t>(b) * kv.Hq + h * G) * kHeadDim;
          __nv_bfloat16 qr[16];  // G <= 16: all loads in flight, then the sum in row order
#pragma unroll
          for (int r = 0; r < 16; ++r)
            qr[r] = r < G ? qg[r * kHeadDim + tid] : __float2bfloat16(0.f);
#pragma unroll
          for (int r = 0; r < 16; ++r)
            if (r < G) qacc += __bfloat162float(qr[r]);
        }
        int ppos[kPB];
#pragma unroll
        for (int i = 0; i < kPB; ++i) {
          const int sl = gid + kPGroups * i;
          ppos[i] = sl < cntP ? P[sl] : -1;
        }
        int cph[kCB];
        float cl[kCB], cvv[kCB];
#pragma unroll
        for (int i = 0; i < kCB; ++i) {
          const int jj = j0 + gid + kPGroups * i;
          cph[i] = jj < j1 && jj < nl ? table[jj] : -1;
          cl[i] = ema1 && gl == 0 && jj < j1 ? ell_r[jj] : 0.f;
          cvv[i] = ema1 && gl == 0 && jj < j1 ? v_r[jj] : 0.f;
        }
        if (tid < kHeadDim) qbar[tid] = qacc / static_cast<float>(G);
        if (tid == 0) {
          s_t0key = 0u;
          s_t1key = 0u;
        }
        named_barrier(1, kPW * 32);
        float qv[16];
        group_query_dims(qbar, gl, qv);

        // ---- wave 2
#pragma unroll
        for (int i = 0; i < kCB; ++i)
          if (cph[i] >= 0 && cph[i] < kv.num_phys)
            stage_record(static_cast<size_t>(cph[i]) * kv.Hkv + h, gid + kPGroups * i);
        int pph[kPB];
#pragma unroll
        for (int i = 0; i < kPB; ++i) {
          const int pos = ppos[i];
          pph[i] = pos >= 0 && pos < nl ? table[pos] : -1;
        }
        float cs[kCB];

        // ---- wave 3 (P_t's records, kPR per group at a time)
#pragma unroll
        for (int i0 = 0; i0 < kPB; i0 += kPR) {
          // warp-uniform: none of the warp's slots left
          if (i0 > 0 && warp * 4 + kPGroups * i0 >= cntP) break;
          uint4 rp[kPR][4];
          float pl[kPR], pv[kPR];  // the old EMA state of those pages
#pragma unroll
          for (int u = 0; u < kPR; ++u) {
            const int pos = ppos[i0 + u];
            if (pph[i0 + u] >= 0 && pph[i0 + u] < kv.num_phys)
              load_record(a.meta, static_cast<size_t>(pph[i0 + u]) * kv.Hkv + h, gl, rp[u]);
            pl[u] = ema1 && gl == 0 && pos >= 0 && pos < n ? ell_r[pos] : 0.f;
            pv[u] = ema1 && gl == 0 && pos >= 0 && pos < n ? v_r[pos] : 0.f;
          }
          if (i0 == 0) {  // the chunk's scores while P_t's first records are in flight
            cp_async_wait_all();
#pragma unroll
            for (int i = 0; i < kCB; ++i) {
              const bool ok = cph[i] >= 0 && cph[i] < kv.num_phys;
              uint4 rc[4];
              if (ok) staged_record(gid + kPGroups * i, rc);
              cs[i] = group_sum(ok ? record_partial<DSA_META_MINMAX>(rc, qv) : 0.f);
            }
          }
#pragma unroll
          for (int u = 0; u < kPR; ++u) {
            const int i = i0 + u, sl = gid + kPGroups * i;
            const bool ok = pph[i] >= 0 && pph[i] < kv.num_phys;
            const float sp = group_sum(ok ? record_partial<DSA_META_MINMAX>(rp[u], qv) : 0.f);
            if (gl == 0 && sl < cntP) {
              spk[sl] = ok ? score_key(sp) : 0u;
              if (ema1) {
                uint32_t key = 0u;
                if (ppos[i] >= 0 && ppos[i] < n) {
                  float l_new, v_new;
                  ema_step(ok ? sp : -INFINITY, pl[u], pv[u], DSA_EMA_UPDATE, a.alpha, a.beta,
                           l_new, v_new);
                  key = score_key(ema_predict(l_new, v_new, a.gamma));
                }
                ppk[sl] = key;
              }
            }
          }
        }
        named_barrier(1, kPW * 32);
        // T0: the k-th largest true score over P_t's pages.  At least k pages score >= T0, so the
        // pages scoring >= T0 contain A_t: they are appended as candidates while scoring, and the
        // selection after the barrier ranks only them (exactly).  T0' likewise for the predictions
        // and P_{t+1} (from the old EMA state).  A missing bound (fewer than k scored pages in P_t)
        // marks the row's list overflowed, and the selection scans every score.
        // (both ranks in one pass over P_t's keys)
        for (int i = tid; i < cntP; i += kPW * 32) {
          const uint32_t ki = spk[i], pi = ema1 ? ppk[i] : 0u;
          int ge = 0, gp = 0;
          for (int q0 = 0; q0 < cntP; q0 += 8) {
            uint32_t kj[8], pj[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              kj[u] = q0 + u < cntP ? spk[q0 + u] : 0u;
              pj[u] = ema1 && q0 + u < cntP ? ppk[q0 + u] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              ge += kj[u] >= ki;
              gp += pj[u] >= pi;
            }
          }
          if (ki != 0u && ge >= a.k) atomicMax(&s_t0key, ki);
          if (pi != 0u && gp >= a.k_pred) atomicMax(&s_t1key, pi);
        }
        named_barrier(1, kPW * 32);
        const uint32_t t0key = s_t0key;
        const uint32_t t1key = ema1 ? s_t1key : 0u;
        if (tid == 0 && t0key == 0u)
          atomicAdd(a.cand_cnt + row, static_cast<unsigned>(kCandCap + 1));
        if (tid == 0 && ema1 && t1key == 0u)
          atomicAdd(a.cand_cnt2 + row, static_cast<unsigned>(kCandCap + 1));
        const long long stage0 = static_cast<long long>(row) * n - s_beg;  // staging index of j = 0
        // the EMA update of page j with score s (staged until the second barrier); returns the key
        // of the prediction
        auto ema_page = [&](int j, float sc, float l_old, float v_old) -> uint32_t {
          float l_new, v_new;
          ema_step(sc, l_old, v_old, DSA_EMA_UPDATE, a.alpha, a.beta, l_new, v_new);
          const float pr = ema_predict(l_new, v_new, a.gamma);
          const int at = static_cast<int>(stage0 + j);
          st_ell[at] = l_new;
          st_v[at] = v_new;
          st_pred[at] = pr;
          return score_key(pr);
        };
        // A round of kCB scored chunk slots per group (lanes with gl == 0 hold a record's score):
        // the outputs, the EMA updates, and the candidates for A_t and P_{t+1}, appended to the
        // row's lists with one counter update per list for the whole CTA.
        auto finish_round = [&](int jb, const bool (&ok)[kCB], const float (&sc)[kCB],
                                const float (&lo)[kCB], const float (&vo)[kCB]) {
          uint32_t kA[kCB], kP[kCB];
          unsigned bA[kCB], bP[kCB];
          int nA = 0, nP = 0;
#pragma unroll
          for (int i = 0; i < kCB; ++i) {
            const int jj = jb + gid + kPGroups * i;
            const bool mine = gl == 0 && jj < j1;
            const float is = ok[i] ? sc[i] : -INFINITY;
            if (mine) outs[jj] = is;
            kA[i] = ok[i] ? score_key(sc[i]) : 0u;
            kP[i] = ema1 && mine ? ema_page(jj, is, lo[i], vo[i]) : 0u;
            bA[i] =
                __ballot_sync(0xffffffffu, t0key != 0u && mine && kA[i] != 0u && kA[i] >= t0key);
            bP[i] = __ballot_sync(0xffffffffu, t1key != 0u && kP[i] != 0u && kP[i] >= t1key);
            nA += __popc(bA[i]);
            nP += __popc(bP[i]);
          }
          // this warp's places among the CTA's candidates, then the CTA's places in the lists; a
          // local counter is cleared by its reader before the second barrier, so the next round
          // finds it zero
          int wA = 0, wP = 0;
          if (lane == 0) {
            if (nA) wA = static_cast<int>(atomicAdd(&s_cand[0], static_cast<unsigned>(nA)));
            if (nP) wP = static_cast<int>(atomicAdd(&s_cand[1], static_cast<unsigned>(nP)));
          }
          named_barrier(1, kPW * 32);
          if (tid == 0) {
            const unsigned c = s_cand[0];
            if (c) s_cand[2] = atomicAdd(a.cand_cnt + row, c);
            s_cand[0] = 0u;
          } else if (tid == 32) {
            const unsigned c = s_cand[1];
            if (c) s_cand[3] = atomicAdd(a.cand_cnt2 + row, c);
            s_cand[1] = 0u;
          }
          named_barrier(1, kPW * 32);
          const unsigned below = (1u << lane) - 1u;
          unsigned atA = s_cand[2] + static_cast<unsigned>(__shfl_sync(0xffffffffu, wA, 0));
          unsigned atP = s_cand[3] + static_cast<unsigned>(__shfl_sync(0xffffffffu, wP, 0));
#pragma unroll
          for (int i = 0; i < kCB; ++i) {
            const int jj = jb + gid + kPGroups * i;
            const unsigned ra = atA + __popc(bA[i] & below), rp = atP + __popc(bP[i] & below);
            if (((bA[i] >> lane) & 1u) && ra < static_cast<unsigned>(kCandCap))
              a.cand[static_cast<size_t>(row) * kCandCap + ra] = make_uint2(kA[i], jj);
            if (((bP[i] >> lane) & 1u) && rp < static_cast<unsigned>(kCandCap))
              a.cand2[static_cast<size_t>(row) * kCandCap + rp] = make_uint2(kP[i], jj);
            atA += __popc(bA[i]);
            atP += __popc(bP[i]);
          }
        };
        {
          bool bad = false, okv[kCB];
#pragma unroll
          for (int i = 0; i < kCB; ++i) {
            const int jj = j0 + gid + kPGroups * i;
            const bool in = jj < j1 && jj < nl;
            okv[i] = in && cph[i] >= 0 && cph[i] < kv.num_phys;
            bad |= in && !okv[i];
          }
          if (gl == 0 && bad) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
          finish_round(j0, okv, cs, cl, cvv);
        }
        // the rest of a long segment, kCB slots per group per round
        for (int jb = j0 + kScoreRecs; jb < j1; jb += kScoreRecs) {
          int ph[kCB];
          float lo[kCB], vo[kCB];
#pragma unroll
          for (int i = 0; i < kCB; ++i) {
            const int jj = jb + gid + kPGroups * i;
            ph[i] = jj < j1 && jj < nl ? table[jj] : -1;
            lo[i] = ema1 && gl == 0 && jj < j1 ? ell_r[jj] : 0.f;
            vo[i] = ema1 && gl == 0 && jj < j1 ? v_r[jj] : 0.f;
          }
#pragma unroll
          for (int i = 0; i < kCB; ++i)
            if (ph[i] >= 0 && ph[i] < kv.num_phys)
              stage_record(static_cast<size_t>(ph[i]) * kv.Hkv + h, gid + kPGroups * i);
          cp_async_wait_all();
          bool bad = false, okv[kCB];
          float sc[kCB];
#pragma unroll
          for (int i = 0; i < kCB; ++i) {
            const int jj = jb + gid + kPGroups * i;
            const bool in = jj < j1 && jj < nl;
            okv[i] = in && ph[i] >= 0 && ph[i] < kv.num_phys;
            bad |= in && !okv[i];
            uint4 rc[4];
            if (okv[i]) staged_record(gid + kPGroups * i, rc);
            sc[i] = group_sum(okv[i] ? record_partial<DSA_META_MINMAX>(rc, qv) : 0.f);
          }
          if (gl == 0 && bad) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
          finish_round(jb, okv, sc, lo, vo);
        }
      }
    };

    // ---- speculative per-page attention of this CTA's items
    auto spec_items = [&]() {
      for (int j = 0; j < my_items; ++j) {
        const int it = irank + j * item_ctas;
        const int row = it / a.k_pred, slot = it - row * a.k_pred;
        const int b = row / kv.Hkv, h = row % kv.Hkv;
        const int L = request_len(kv, b);
        const int s = j % kPStages;
        named_barrier(1, kPW * 32);  // the previous item's query rows are no longer read
        if (j > 0) stage_q(j);
        cp_async_wait_all();
        named_barrier(1, kPW * 32);
        uint32_t qa[8][4];
        load_q_frags(sQ, qa);
        WarpSoftmaxState st;
        state_init(st);
        const bool got = mbar_wait(smem_u32(&bars[s]), (j / kPStages) & 1, abort_flag, kv.status);
        const int okv = got ? stage_ok[s] : -1;
        const int pos = stage_pos[s];
        if (okv == 1) {
          const uint32_t kb = smem_base + s * stage_bytes;
          const uint32_t vb = kb + 2 * page * 128;
          bool wrote = false;
          for (int t = warp; t < tiles; t += kPW) {
            const bool in = pos * page + t * 16 + (lane & 15) < L;
            const uint32_t vm = __ballot_sync(0xffffffffu, in) & 0xffffu;
            if (vm == 0u) continue;
            if (vm != 0xffffu)
              wrote |=
                  zero_invalid_v_rows(vm, smem + s * stage_bytes + 2 * page * 128, page, t * 16);
            float sc[2][4];
            tile_scores(qa, kb, page, t * 16, sc);
            tile_softmax_pv(st, sc, a.scale_log2, vm, vb, page, t * 16);
          }
          if (wrote) fence_proxy_async_smem();
        }
        __syncwarp();
        if (got && lane == 0) mbar_arrive(smem_u32(&bars[kPStages + s]));
        state_finish(st);
        {
          const int r0 = lane >> 2, c0 = (lane & 3) * 2;
          float* wO = sO + warp * G * kHeadDim;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (r0 < G)
              *reinterpret_cast<float2*>(wO + r0 * kHeadDim + jj * 8 + c0) =
                  make_float2(st.o[jj][0], st.o[jj][1]);
            if (r0 + 8 < G)
              *reinterpret_cast<float2*>(wO + (r0 + 8) * kHeadDim + jj * 8 + c0) =
                  make_float2(st.o[jj][2], st.o[jj][3]);
          }
          if ((lane & 3) == 0) {
            if (r0 < G) {
              sM[warp * G + r0] = st.m[0];
              sL[warp * G + r0] = st.l[0];
            }
            if (r0 + 8 < G) {
              sM[warp * G + r0 + 8] = st.m[1];
              sL[warp * G + r0 + 8] = st.l[1];
            }
          }
        }
        // a wait that gave up in any consumer warp makes every warp skip the record (the OR over
        // the barrier is the same in all of them), so the barrier inside stays uniform
        const bool gave_up = named_barrier_or(1, kPW * 32, !got || *abort_flag);
        if (okv >= 0 && !gave_up) {
          float* rec0 =
              a.partials + (static_cast<size_t>(row) * a.k_pred + slot) * G * kRecordFloats;
          if (okv == 0) {  // a position outside the request: the empty part
            for (int g = tid; g < G; g += kPW * 32)
              *reinterpret_cast<float4*>(rec0 + g * kRecordFloats + 128) =
                  make_float4(-INFINITY, 0.f, 0.f, 0.f);
          } else {
            // per head: the warps' weights exp(m_w - M) / l (one division each) and the record's
            // (m, l); then O = sum_w weight_w O_w as float4 rows
            const int nwu = min(tiles, kPW);  // warps that attended a tile
            if (tid < G) {
              const int g = tid;
              float M = -INFINITY;
              for (int w = 0; w < nwu; ++w) M = fmaxf(M, sM[w * G + g]);
              float Lsum = 0.f;
              for (int w = 0; w < nwu; ++w) {
                const float mw = sM[w * G + g];
                const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                wt[w * 16 + g] = f;
                Lsum += sL[w * G + g] * f;
              }
              const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
              for (int w = 0; w < nwu; ++w) wt[w * 16 + g] *= inv;
              *reinterpret_cast<float4*>(rec0 + g * kRecordFloats + 128) =
                  make_float4(M == -INFINITY ? -INFINITY : M * kLn2, Lsum, 0.f, 0.f);
            }
            named_barrier(1, kPW * 32);
            for (int e = tid; e < G * 32; e += kPW * 32) {
              const int g = e >> 5, d4 = e & 31;
              float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int w = 0; w < nwu; ++w) {
                const float f = wt[w * 16 + g];
                const float4 o =
                    *reinterpret_cast<const float4*>(sO + (w * G + g) * kHeadDim + d4 * 4);
                acc.x = fmaf(f, o.x, acc.x);
                acc.y = fmaf(f, o.y, acc.y);
                acc.z = fmaf(f, o.z, acc.z);
                acc.w = fmaf(f, o.w, acc.w);
              }
              *reinterpret_cast<float4*>(rec0 + g * kRecordFloats + d4 * 4) = acc;
            }
          }
        }
      }
    };
    score_share();
    spec_items();
  }
  // addresses a role reads first after the barrier
  if (tid == 0 && roles) {
    if (p_role) {
      const int row = cta - rows;
      prefetch_l2(a.cand_cnt2 + row);
      prefetch_l2(a.cand2 + static_cast<size_t>(row) * kCandCap);
      prefetch_l2(a.next_idx + static_cast<size_t>(row) * a.k_pred);
      prefetch_l2(a.next_count + row);
    } else if (rep_first < rows * G) {
      const int row = rep_first / G;
      prefetch_l2(a.cand_cnt + row);
      prefetch_l2(a.cand + static_cast<size_t>(row) * kCandCap);
    }
  }
  grid_arrive(a.sync + 0, abort_flag);
  if (!rehearse && !grid_wait(a.sync + 0, gridDim.x, abort_flag, kv.status)) {
    // gave up: wait (bounded) for this CTA's page loads still in flight before exiting
    if (tid == 0) {
      const int n_iss = *reinterpret_cast<volatile int*>(&s_issued);
      for (int j = max(0, n_iss - kPStages); j < n_iss; ++j) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(smem_u32(&bars[j % kPStages]), (j / kPStages) & 1))
          if (global_timer_ns() - t0 > 50000000ull) break;
      }
    }
    return;
  }

  // ================================================================ phase 2
  // With the roles, CTAs [rows, 2 rows) select P_{t+1} (and update the EMA unless scoring did),
  // which only the next step reads, beside the repair.  Rows are read as float4, four per thread
  // in flight.
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + lay.keys_off);
  const bool vec4 = (n & 3) == 0 &&
                    ((reinterpret_cast<uintptr_t>(a.scores) | reinterpret_cast<uintptr_t>(a.ell) |
                      reinterpret_cast<uintptr_t>(a.trend) |
                      reinterpret_cast<uintptr_t>(a.pred)) & 15) == 0;
  // Without the roles (2 rows CTAs or fewer) everyone selects A_t of its rows, waits, then
  // updates the EMA and repairs.
  auto select_into = [&](int kk, int32_t* out, int32_t* cnt, KeyStats st) {
    __syncthreads();
    const int total = select_topk_block<kPThreads>(keys, n, kk, out, sel_scratch, st);
    if (tid == 0) *cnt = total;
  };
  // P_{t+1} = top-k_pred of the prediction.  Speculated like A_t: the k_pred-th largest predicted
  // score over P_t's pages bounds it from below, so the pages predicted at or above that bound are
  // collected while the EMA state is updated, and only they are ranked (the whole row falls back
  // to the full selection when P_t has fewer than k_pred scored pages or too many pages pass).
  TopkScratch& ts = sel_scratch.small;
  unsigned* pkeys = reinterpret_cast<unsigned*>(ts.crank);  // predicted keys of P_t's pages
  auto ema_row = [&](int row) {
    const size_t base = static_cast<size_t>(row) * n;
    KeyStats st;
    __syncthreads();  // keys / scratch of a previous task are no longer read
    const int cntP = min(max(a.spec_count[row], 0), a.k_pred);
    const int32_t* P = a.spec_idx + static_cast<size_t>(row) * a.k_pred;
    if (tid == 0) {
      s_t0key = 0u;
      ts.n_cand = 0;
    }
    for (int i = tid; i < cntP; i += kPThreads) {
      const int p = P[i];
      uint32_t key = 0u;
      if (p >= 0 && p < n) {
        float l_new, v_new;
        ema_step(__ldcg(a.scores + base + p), a.ell[base + p], a.trend[base + p], DSA_EMA_UPDATE,
                 a.alpha, a.beta, l_new, v_new);
        key = score_key(ema_predict(l_new, v_new, a.gamma));
      }
      pkeys[i] = key;
    }
    __syncthreads();
    for (int i = tid; i < cntP; i += kPThreads) {
      const uint32_t ki = pkeys[i];
      if (ki == 0u) continue;
      int ge = 0;
      for (int j0 = 0; j0 < cntP; j0 += 8) {
        uint32_t kj[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) kj[u] = j0 + u < cntP ? pkeys[j0 + u] : 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u) ge += kj[u] >= ki;
      }
      if (ge >= a.k_pred) atomicMax(&s_t0key, ki);
    }
    __syncthreads();
    const uint32_t t0 = s_t0key;
    // predicted keys >= t0 become candidates (one shared counter update per warp)
    auto collect = [&](int j, uint32_t key) {
      const bool c = t0 != 0u && key != 0u && key >= t0;
      const unsigned bal = __ballot_sync(0xffffffffu, c);
      if (bal == 0u) return;
      int at0 = 0;
      if (lane == 0) at0 = atomicAdd(&ts.n_cand, __popc(bal));
      at0 = __shfl_sync(0xffffffffu, at0, 0);
      const int at = at0 + __popc(bal & ((1u << lane) - 1u));
      if (c && at < kTopkMaxCand) {
        ts.ckey[at] = key;
        ts.cidx[at] = j;
      }
    };
    if (vec4) {
      const int n4 = n >> 2;
      for (int i0 = tid; i0 < ((n4 + 31) & ~31); i0 += 2 * kPThreads) {
        float4 is[2], lo[2], vo[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = i0 + u * kPThreads;
          if (i < n4) {
            is[u] = __ldcg(reinterpret_cast<const float4*>(a.scores + base) + i);
            lo[u] = *(reinterpret_cast<const float4*>(a.ell + base) + i);
            vo[u] = *(reinterpret_cast<const float4*>(a.trend + base) + i);
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = i0 + u * kPThreads;
          uint32_t kq[4] = {0u, 0u, 0u, 0u};
          if (i < n4) {
            float4 ln, vn, pr;
            ema_step(is[u].x, lo[u].x, vo[u].x, DSA_EMA_UPDATE, a.alpha, a.beta, ln.x, vn.x);
            ema_step(is[u].y, lo[u].y, vo[u].y, DSA_EMA_UPDATE, a.alpha, a.beta, ln.y, vn.y);
            ema_step(is[u].z, lo[u].z, vo[u].z, DSA_EMA_UPDATE, a.alpha, a.beta, ln.z, vn.z);
            ema_step(is[u].w, lo[u].w, vo[u].w, DSA_EMA_UPDATE, a.alpha, a.beta, ln.w, vn.w);
            pr.x = ema_predict(ln.x, vn.x, a.gamma);
            pr.y = ema_predict(ln.y, vn.y, a.gamma);
            pr.z = ema_predict(ln.z, vn.z, a.gamma);
            pr.w = ema_predict(ln.w, vn.w, a.gamma);
            *(reinterpret_cast<float4*>(a.ell + base) + i) = ln;
            *(reinterpret_cast<float4*>(a.trend + base) + i) = vn;
            if (a.pred) *(reinterpret_cast<float4*>(a.pred + base) + i) = pr;
            kq[0] = score_key(pr.x);
            kq[1] = score_key(pr.y);
            kq[2] = score_key(pr.z);
            kq[3] = score_key(pr.w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              keys[4 * i + e] = kq[e];
              st.add(kq[e]);
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) collect(4 * i + e, kq[e]);
        }
      }
    } else {
      for (int j0 = tid; j0 < ((n + 31) & ~31); j0 += kPThreads) {
        uint32_t key = 0u;
        if (j0 < n) {
          float l_new, v_new;
          ema_step(__ldcg(a.scores + base + j0), a.ell[base + j0], a.trend[base + j0],
                   DSA_EMA_UPDATE, a.alpha, a.beta, l_new, v_new);
          a.ell[base + j0] = l_new;
          a.trend[base + j0] = v_new;
          const float p = ema_predict(l_new, v_new, a.gamma);
          if (a.pred) a.pred[base + j0] = p;
          key = score_key(p);
          keys[j0] = key;
          st.add(key);
        }
        collect(j0, key);
      }
    }
    __syncthreads();
    int32_t* out = a.next_idx + static_cast<size_t>(row) * a.k_pred;
    const int C = ts.n_cand;
    if (t0 != 0u && C <= kTopkMaxCand) {
      const int total = topk_candidates<kPThreads>(C, a.k_pred, n, out, ts);
      for (int i = total + tid; i < a.k_pred; i += kPThreads) out[i] = -1;
      if (tid == 0) a.next_count[row] = total;
    } else {
      select_into(a.k_pred, out, a.next_count + row, st);
    }
  };
  // A_t of a row into out[0, k) (ascending, -1 past the count); returns the count.  The top-k of
  // the candidates that scored at or above T0 (exact, see scoring), else of the whole row.
  // `side` is work that overlaps the ranking (after it in the whole-row case, whose keys share the
  // record area).
  auto select_a = [&](int row, int32_t* out, auto&& side) -> int {
    const size_t base = static_cast<size_t>(row) * n;
    __syncthreads();  // keys / scratch of a previous task are no longer read
    // the list up to its capacity is read together with its count (one round trip); the entries
    // below the count index pages < n, and the clamp keeps a rehearsal, which reads the list while
    // it is still being appended to, inside the bitmap
    unsigned C = __ldcg(a.cand_cnt + row);
    // a rehearsal ranks at least 2k entries (whatever the list holds), so that code runs
    if (dry) C = min(max(C, static_cast<unsigned>(2 * a.k)), static_cast<unsigned>(kCandCap));
    {
      const uint2* cr = a.cand + static_cast<size_t>(row) * kCandCap;
      for (int i = tid; i < kCandCap; i += kPThreads) {
        const uint2 e = __ldcg(cr + i);
        ts.ckey[i] = e.x;
        ts.cidx[i] = static_cast<int>(min(e.y, static_cast<unsigned>(n - 1)));
      }
    }
    if (C <= static_cast<unsigned>(kCandCap)) {
      side();
      __syncthreads();
      const int total = topk_candidates<kPThreads>(static_cast<int>(C), a.k, n, out, ts);
      for (int i = total + tid; i < a.k; i += kPThreads) out[i] = -1;
      return total;
    }
    KeyStats st;
    if (vec4) {
      const int n4 = n >> 2;
      for (int i0 = tid; i0 < n4; i0 += 8 * kPThreads) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * kPThreads;
          if (i < n4) v[u] = __ldcg(reinterpret_cast<const float4*>(a.scores + base) + i);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * kPThreads;
          if (i >= n4) continue;
          keys[4 * i + 0] = score_key(v[u].x);
          keys[4 * i + 1] = score_key(v[u].y);
          keys[4 * i + 2] = score_key(v[u].z);
          keys[4 * i + 3] = score_key(v[u].w);
          st.add(keys[4 * i + 0]);
          st.add(keys[4 * i + 1]);
          st.add(keys[4 * i + 2]);
          st.add(keys[4 * i + 3]);
        }
      }
    } else {
      for (int j = tid; j < n; j += kPThreads) {
        keys[j] = score_key(__ldcg(a.scores + base + j));
        st.add(keys[j]);
      }
    }
    __syncthreads();
    const int total = select_topk_block<kPThreads>(keys, n, a.k, out, sel_scratch, st);
    __syncthreads();  // the keys are no longer read
    side();
    return total;
  };
  // membership bitmaps over page positions [0, n): P_t's and A_t's
  const int bm_words = (n + 31) >> 5;
  // a repair task's lists: P_t (positions and bitmap), the query head; A_t's bitmap cleared
  auto fetch_lists = [&](int task) {
    int32_t* sP = reinterpret_cast<int32_t*>(smem + lay.sp_off);
    float* qh = reinterpret_cast<float*>(smem + lay.qh_off);
    uint32_t* bmP = reinterpret_cast<uint32_t*>(smem + lay.bmp_off);
    uint32_t* bmA = reinterpret_cast<uint32_t*>(smem + lay.bma_off);
    const int row = task / G, g = task - row * G;
    const int b = row / kv.Hkv, h = row % kv.Hkv;
    const int cntP = min(max(a.spec_count[row], 0), a.k_pred);
    for (int w = tid; w < bm_words; w += kPThreads) {
      bmP[w] = 0u;
      bmA[w] = 0u;
    }
    const size_t qhead = static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G + g;
    for (int d = tid; d < kHeadDim; d += kPThreads)
      qh[d] = __bfloat162float(a.q[qhead * kHeadDim + d]) * a.scale_log2;
    __syncthreads();
    for (int i = tid; i < cntP; i += kPThreads) {
      const int pos = a.spec_idx[static_cast<size_t>(row) * a.k_pred + i];
      sP[i] = pos;
      if (pos >= 0 && pos < n) atomicOr(&bmP[pos >> 5], 1u << (pos & 31));
    }
  };
  // the speculative records of a task's query head (phase 1 wrote them before the first
  // barrier), copied asynchronously into shared memory: complete after cp_async_wait_all
  auto fetch_records = [&](int task) {
    const int row = task / G, g = task - row * G;
    const int cntP = min(max(a.spec_count[row], 0), a.k_pred);
    const uint32_t srec = smem_u32(smem + lay.rec_off);
    constexpr int kPieces = kRecordFloats / 4;  // 16-byte pieces of a record
    for (int e = tid; e < cntP * kPieces; e += kPThreads) {
      const int i = e / kPieces, c = e - i * kPieces;
      cp_async16(srec + static_cast<uint32_t>(i * kRecordFloats + c * 4) * 4u,
                 a.partials + ((static_cast<size_t>(row) * a.k_pred + i) * G + g) * kRecordFloats +
                     c * 4);
    }
  };

  // P_{t+1} of a row whose EMA update rode along with scoring: rank the candidates, or (no
  // bound, or too many candidates) recompute the row's predictions from the old state, which is
  // only overwritten after the second barrier, and select from all of them
  auto next_row = [&](int row) {
    const size_t base = static_cast<size_t>(row) * n;
    __syncthreads();  // keys / scratch of a previous task are no longer read
    int32_t* out = a.next_idx + static_cast<size_t>(row) * a.k_pred;
    const unsigned C = __ldcg(a.cand_cnt2 + row);
    {
      const uint2* cr = a.cand2 + static_cast<size_t>(row) * kCandCap;
      for (int i = tid; i < kCandCap; i += kPThreads) {
        const uint2 e = __ldcg(cr + i);
        ts.ckey[i] = e.x;
        ts.cidx[i] = static_cast<int>(min(e.y, static_cast<unsigned>(n - 1)));
      }
    }
    if (C <= static_cast<unsigned>(kCandCap)) {
      __syncthreads();
      const int total = topk_candidates<kPThreads>(static_cast<int>(C), a.k_pred, n, out, ts);
      for (int i = total + tid; i < a.k_pred; i += kPThreads) out[i] = -1;
      if (tid == 0) a.next_count[row] = total;
      return;
    }
    KeyStats st;
    for (int j = tid; j < n; j += kPThreads) {
      float l_new, v_new;
      ema_step(__ldcg(a.scores + base + j), a.ell[base + j], a.trend[base + j], DSA_EMA_UPDATE,
               a.alpha, a.beta, l_new, v_new);
      keys[j] = score_key(ema_predict(l_new, v_new, a.gamma));
      st.add(keys[j]);
    }
    select_into(a.k_pred, out, a.next_count + row, st);
  };
  if (p_role) {
    if (ema1) next_row(cta - rows);
    else ema_row(cta - rows);
    // counts the P_{t+1} CTAs past their reads of the old EMA state (the staged updates wait
    // for all of them)
    grid_arrive(a.sync + 1, abort_flag);
  } else if (!roles) {
    for (int row = cta; row < rows; row += grid) {
      const int total = select_a(row, a.idx + static_cast<size_t>(row) * a.k, [] {});
      if (tid == 0) a.count[row] = total;
    }
    if (!grid_barrier(a.sync + 1, gridDim.x, abort_flag, kv.status)) return;
    for (int row = cta; row < rows; row += grid) ema_row(row);
  }

  // ================================================================ phase 3
  // per (row, query head): attention over the missed pages A_t \ P_t on the CUDA cores, merged
  // with the speculative records of A_t ∩ P_t (every record of P_t in superset mode).  Each warp
  // keeps one online-softmax state (log2 units, unnormalised O) over its missed tokens and its
  // share of the records; the nine states are combined at the end.
  int32_t* sP = reinterpret_cast<int32_t*>(smem + lay.sp_off);
  int32_t* sA = reinterpret_cast<int32_t*>(smem + lay.sa_off);
  int2* list = reinterpret_cast<int2*>(smem + lay.list_off);         // missed (phys, pos)
  int32_t* parts = reinterpret_cast<int32_t*>(smem + lay.part_off);  // merged P slots
  float* qh = reinterpret_cast<float*>(smem + lay.qh_off);
  float* wst = reinterpret_cast<float*>(smem + lay.ws_off);  // [warp][m, l, -, -, O[128]]
  constexpr int kWs = kHeadDim + 4;
  const int task0 = dry ? (cta / kScoutEvery) % (rows * G) : rep_first;
  const int task_step = dry ? rows * G : rep_step;
  for (int task = task0; task >= 0 && task < rows * G; task += task_step) {
    const int row = task / G, g = task - row * G;
    const int b = row / kv.Hkv, h = row % kv.Hkv;
    const int L = request_len(kv, b);
    const int npos = (L + page - 1) / page;
    const size_t qhead = static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G + g;
    const int cntP = min(max(a.spec_count[row], 0), a.k_pred);
    __syncthreads();  // shared lists of a previous task are no longer read
    fetch_lists(task);
    uint32_t* bmP = reinterpret_cast<uint32_t*>(smem + lay.bmp_off);
    uint32_t* bmA = reinterpret_cast<uint32_t*>(smem + lay.bma_off);
    int cntA;
    if (roles) {
      cntA = select_a(row, sA, [&] { fetch_records(task); });
      __syncthreads();  // sA is complete
      if (g == 0 && !dry) {  // the task of the row's first query head publishes A_t
        for (int i = tid; i < a.k; i += kPThreads)
          a.idx[static_cast<size_t>(row) * a.k + i] = sA[i];
        if (tid == 0) a.count[row] = cntA;
      }
    } else {
      fetch_records(task);
      // the whole index row at once (slots past the count hold -1), together with the count
      cntA = __ldcg(a.count + row);
      for (int i = tid; i < a.k; i += kPThreads)
        sA[i] = __ldcg(a.idx + static_cast<size_t>(row) * a.k + i);
      __syncthreads();
    }
    cntA = min(max(cntA, 0), a.k);
    for (int i = tid; i < cntA; i += kPThreads) {
      const int pos = sA[i];
      if (pos >= 0 && pos < n) atomicOr(&bmA[pos >> 5], 1u << (pos & 31));
    }
    cp_async_wait_all();  // this thread's record pieces
    __syncthreads();
    auto in_bm = [&](const uint32_t* bm, int pos) {
      return pos >= 0 && pos < n && ((bm[pos >> 5] >> (pos & 31)) & 1u);
    };
    // merged speculative parts (warp 0): P slots whose page is in A (every slot in superset
    // mode); missed pages (warp 1): A \ P inside the request with a valid page-table entry
    if (warp == 0) {
      int np = 0;
      for (int base = 0; base < cntP; base += 32) {
        const int i = base + lane;
        const bool take = i < cntP && (a.superset || in_bm(bmA, sP[i]));
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        if (take) parts[np + __popc(bal & ((1u << lane) - 1u))] = i;
        np += __popc(bal);
      }
      if (lane == 0) s_red[0] = np;
    } else if (warp == 1) {
      int nm = 0;
      for (int base = 0; base < cntA; base += 32) {
        const int i = base + lane;
        int phys = 0, pos = -1;
        bool miss = false;
        if (i < cntA) {
          pos = sA[i];
          miss = !in_bm(bmP, pos) && lookup_page(kv, b, pos, npos, &phys);
        }
        const unsigned bal = __ballot_sync(0xffffffffu, miss);
        if (miss) list[nm + __popc(bal & ((1u << lane) - 1u))] = make_int2(phys, pos);
        nm += __popc(bal);
      }
      if (lane == 0) s_red[1] = nm;
    }
    __syncthreads();
    const int n_parts = s_red[0];
    const int n_miss = dry ? min(s_red[1], 1) : s_red[1];  // a rehearsal attends one page at most

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
    // ---- missed tokens, 32 per warp round (lane = token for q.k, lane = 4 dims for p.v); the
    // round's V rows are requested together with its K rows
    const int cpp = (page + 31) / 32;  // 32-token chunks per page
    for (int c = warp; c < n_miss * cpp; c += kPWarps) {
      const int pi = c / cpp, sub = c - pi * cpp;
      const int phys = list[pi].x, pos = list[pi].y;
      const int t0 = sub * 32;  // first slot of the chunk within the page
      const int nvalid = max(0, min(min(32, page - t0), L - (pos * page + t0)));
      const size_t row0 = (static_cast<size_t>(phys) * kv.Hkv + h) * page + t0;
      const __nv_bfloat16* vrow = a.vpool + row0 * kHeadDim + lane * 4;
      uint2 vr[32];
#pragma unroll
      for (int u = 0; u < 32; ++u)
        vr[u] = u < nvalid ? __ldg(reinterpret_cast<const uint2*>(vrow + static_cast<size_t>(u) *
                                                                                kHeadDim))
                           : make_uint2(0u, 0u);
      float s = -INFINITY;
      if (lane < nvalid) {
        const uint4* kr = reinterpret_cast<const uint4*>(a.kpool + (row0 + lane) * kHeadDim);
        float acc = 0.f;
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          uint4 raw[8];
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) raw[c8] = __ldg(kr + h8 * 8 + c8);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&raw[c8]);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              acc = fmaf(qh[(h8 * 8 + c8) * 8 + e], __bfloat162float(v[e]), acc);
          }
        }
        s = acc;
      }
      const float cmax = warp_max(s);
      if (cmax == -INFINITY) continue;
      const float p = lane < nvalid ? fast_exp2(s - cmax) : 0.f;
      const float lsum = warp_sum(p);
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const float pt = __shfl_sync(0xffffffffu, p, u);
        const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&vr[u]);
        o.x = fmaf(pt, __bfloat162float(v[0]), o.x);
        o.y = fmaf(pt, __bfloat162float(v[1]), o.y);
        o.z = fmaf(pt, __bfloat162float(v[2]), o.z);
        o.w = fmaf(pt, __bfloat162float(v[3]), o.w);
      }
      const float inv = 1.f / lsum;
      absorb(cmax, lsum, make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv));
    }
    // ---- speculative records (prefetched to shared memory), eight per warp round
    for (int i0 = warp; i0 < n_parts; i0 += 8 * kPWarps) {
      float mv[8], lv[8];
      float4 ov[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kPWarps;
        mv[u] = -INFINITY;
        lv[u] = 0.f;
        ov[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < n_parts) {
          const float* r =
              reinterpret_cast<const float*>(smem + lay.rec_off) + parts[i] * kRecordFloats;
          mv[u] = r[128];
          lv[u] = r[129];
          ov[u] = *(reinterpret_cast<const float4*>(r) + lane);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) absorb(mv[u] * kLog2e, lv[u], ov[u]);
    }
    if (lane == 0) {
      wst[warp * kWs] = wm;
      wst[warp * kWs + 1] = wl;
    }
    *reinterpret_cast<float4*>(wst + warp * kWs + 4 + lane * 4) = wo;
    __syncthreads();
    // ---- combine the warps' states
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kPWarps; ++w)
      if (wst[w * kWs + 1] > 0.f) M = fmaxf(M, wst[w * kWs]);
    if (tid < kHeadDim) {
      float o = 0.f, lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kPWarps; ++w) {
        const float lw = wst[w * kWs + 1];
        if (!(lw > 0.f)) continue;
        const float f = fast_exp2(wst[w * kWs] - M);
        lsum += lw * f;
        o += wst[w * kWs + 4 + tid] * f;
      }
      const float ov = lsum > 0.f ? o / lsum : 0.f;
      if (!dry) a.out[qhead * kHeadDim + tid] = ov;
      if (tid == 0 && !dry) {
        a.m[qhead] = lsum > 0.f ? M * kLn2 : -INFINITY;
        a.l[qhead] = lsum;
      }
    }
  }

  if (ema1) {
    // the staged EMA updates of this CTA's share, once every P_{t+1} CTA is past its reads of
    // the old state
    if (!grid_wait(a.sync + 1, rows, abort_flag, kv.status)) return;
    const int cnt = static_cast<int>(s_end - s_beg);
    for (int i = tid; i < cnt; i += kPThreads) {
      a.ell[s_beg + i] = st_ell[i];
      a.trend[s_beg + i] = st_v[i];
      if (a.pred) a.pred[s_beg + i] = st_pred[i];
    }
  }

  // ---- the last CTA out resets the barrier counters for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sync + 2, 1u) == gridDim.x - 1) {
      for (int r = 0; r < rows; ++r) {
        a.cand_cnt[r] = 0u;
        a.cand_cnt2[r] = 0u;
      }
      a.sync[0] = 0u;
      a.sync[1] = 0u;
      a.sync[2] = 0u;
      __threadfence();
    }
  }
}

}  // namespace

size_t prr_step_workspace_bytes(int rows) {
  const size_t cnt = (4 * static_cast<size_t>(rows) + 15) & ~static_cast<size_t>(15);
  const size_t list = static_cast<size_t>(rows) * kCandCap * sizeof(uint2);
  return 256 + 2 * (cnt + list);
}

size_t prr_step_smem_bytes(int page, int G, int n, int k, int k_pred) {
  return playout(page, G, n, k, k_pred).total;
}

cudaError_t launch_prr_step(const CUtensorMap& tmK, const CUtensorMap& tmV, const PrrStepArgs& s,
                            cudaStream_t stream) {
  PrrArgs a;
  a.kv = s.kv;
  a.kpool = s.kpool;
  a.vpool = s.vpool;
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
  a.sync = s.sync;
  a.cand_cnt = s.cand_cnt;
  a.cand = s.cand;
  a.cand_cnt2 = s.cand_cnt2;
  a.cand2 = s.cand2;
  const size_t bytes = playout(s.kv.p, s.kv.G, s.stride, s.k, s.k_pred).total;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(prr_step_kernel), bytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prr_step_kernel, kPThreads,
                                                         bytes)) != cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // every CTA must be resident at once (the phases wait on each other): a cooperative launch
  // of one CTA per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prr_step_kernel, tmK, tmV, a);
}

}  // namespace dsa
