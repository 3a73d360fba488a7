// Shared device helpers for libdsa (sm_103a): PTX wrappers for mbarriers, TMA tile loads,
// ldmatrix and bf16 mma, bounded waits, order-preserving float keys and block reductions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"
#include "internal.h"

#define DSA_DEV __device__ __forceinline__

namespace dsa {

// Bounded waits give up after this many nanoseconds and raise DSA_STATUS_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

DSA_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared memory window advanced to a 1024-byte boundary (the 128-byte TMA swizzle
// pattern repeats every 1024 bytes), as an offset from the __shared__ array itself so that every
// pointer derived from it stays in the shared address space (a detour through an integer would
// turn its accesses into generic ones).
DSA_DEV uint8_t* smem_align1024(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

DSA_DEV unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

DSA_DEV void raise_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Tokens of request b, clamped to what its page-table row can address.
DSA_DEV int request_len(const KvView& kv, int b) {
  return min(max(kv.seq_lens[b], 0), kv.p * kv.max_pages);
}

// ------------------------------------------------------------------------------- mbarrier

DSA_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

DSA_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

DSA_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// Adds `bytes` to the transaction count of the barrier's current phase without arriving (several
// threads may each post the bytes of the copies they issue; one arrival then closes the phase).
DSA_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

DSA_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The waiting thread is suspended until the phase completes or kWaitSuspendNs pass, so that a
// waiting warp does not spin on issue slots its SM sub-partition's working warps need.
constexpr uint32_t kWaitSuspendNs = 100000;

DSA_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kWaitSuspendNs)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after kWaitLimitNs, raising
// DSA_STATUS_TIMEOUT and setting *abort so that the rest of the CTA stops waiting too.
DSA_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (*abort) return false;
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      raise_status(status, DSA_STATUS_TIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------------------------------------- TMA

// One KV page (both 64-dim halves of `page` token rows) global -> shared with one 3-D tiled
// bulk tensor load completing on an mbarrier (complete_tx::bytes).  The pool's tensor map views it
// as (64 dims, token rows, 2 halves) with box (64, page, 2) and 128-byte swizzle, so the page
// lands as dims 0..63 of every row followed by dims 64..127 of every row, each line 128 bytes.
DSA_DEV void tma_load_page(uint32_t dst, const CUtensorMap* map, int row0, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row0), "r"(0), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16), completing on
// an mbarrier.
DSA_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// 16-byte asynchronous global -> shared copy through L2 (no register staging); completed for the
// issuing thread by cp_async_wait_all.
DSA_DEV void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

DSA_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Named barrier over `count` threads (a multiple of 32) of the CTA.
DSA_DEV void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialization may
// start while the kernel before it in the stream is still running: it runs only set-up that
// touches no global memory written by earlier work, then waits here until every prerequisite
// grid has completed and its memory operations are visible.  Without such a dependency the wait
// returns at once.
DSA_DEV void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the kernel that follows in the stream be scheduled before this one completes (its blocks
// take SMs as this kernel's blocks leave them, and wait at grid_dependency_wait).
DSA_DEV void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Arrival at a named barrier without waiting (the arriving threads' earlier shared-memory writes
// are visible to the threads that wait at it).
DSA_DEV void named_barrier_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also returns the OR of a predicate over the participating threads (the same
// value in every thread).
DSA_DEV bool named_barrier_or(int id, int count, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

// Prefetches the line holding p into L2; issued early, it also brings the page's address
// translation in before the data is needed.  Never waits.
DSA_DEV void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

DSA_DEV void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) access.
DSA_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of 128-byte line `line` in a tile written by TMA
// with CU_TENSOR_MAP_SWIZZLE_128B (tile base 1024-byte aligned).
DSA_DEV uint32_t sw128(uint32_t line, uint32_t chunk) {
  return line * 128u + ((chunk ^ (line & 7u)) << 4);
}

// ------------------------------------------------------------------------------- tensor core

DSA_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

DSA_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A (16x16 bf16, row) * B (16x8 bf16, col) + D, fp32 accumulate.
DSA_DEV void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

DSA_DEV uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x via the SFU instruction (approximate; relative error far below the bf16 rounding of P).
DSA_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) via the SFU instruction (approximate: absolute error about 2^-22 on [0.5, 2], relative
// elsewhere; lg2(0) = -inf).
DSA_DEV float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------------------- keys

// Order-preserving map of a float score to uint32 (larger score -> larger key, equal scores ->
// equal keys).  Entries that are not candidates (-inf, NaN) map to 0; every other float maps to a
// key >= 0x00800000.
DSA_DEV uint32_t score_key(float s) {
  if (!(s > -INFINITY)) return 0u;
  uint32_t b = s == 0.f ? 0u : __float_as_uint(s);  // -0 and +0 are the same score
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ------------------------------------------------------------------------------- reductions

DSA_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

DSA_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

DSA_DEV int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Exclusive prefix sum over the block (blockDim.x a multiple of 32, <= 1024).  `scratch` holds
// 33 ints.  Returns this thread's exclusive prefix; *total receives the block total.
DSA_DEV int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;  // inclusive over warps
    if (lane == 31) scratch[32] = w;
  }
  __syncthreads();
  const int base = warp > 0 ? scratch[warp - 1] : 0;
  const int res = base + x - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// ------------------------------------------------------------------------------- phase tracing

// A library built with -DDSA_TIMELINE (libdsa_trace.so, never libdsa.so) records, for thread 0 of
// each of the first kTraceCtas CTAs of an instrumented kernel, clock64() and %globaltimer the
// first time it passes each numbered stamp: DSA_TRACE_BEGIN() at the kernel's start (a barrier
// and stamp 0), DSA_STAMP(k) at a phase boundary, DSA_TRACE_END(store) where every thread of the
// CTA meets at the end.  The stamps are ordered against the surrounding code only as volatile
// operations are, so they bound phases approximately.  Built without the define, all three expand
// to nothing.
constexpr int kTraceCtas = 1024, kTraceSlots = 32;
#ifdef DSA_TIMELINE
#define DSA_TRACE_BEGIN()                                              \
  __shared__ unsigned long long s_trace_[2 * ::dsa::kTraceSlots];      \
  if (threadIdx.x < 2 * ::dsa::kTraceSlots) s_trace_[threadIdx.x] = 0; \
  __syncthreads();                                                     \
  DSA_STAMP(0)
#define DSA_STAMP(k)                                                     \
  do {                                                                   \
    if (threadIdx.x == 0 && s_trace_[k] == 0ull) {                       \
      s_trace_[k] = clock64();                                           \
      s_trace_[::dsa::kTraceSlots + (k)] = ::dsa::global_timer_ns();     \
    }                                                                    \
  } while (0)
#define DSA_TRACE_END(store)                                                         \
  do {                                                                               \
    __syncthreads();                                                                 \
    if (threadIdx.x < 2 * ::dsa::kTraceSlots && blockIdx.x < ::dsa::kTraceCtas)      \
      (store)[blockIdx.x * 2 * ::dsa::kTraceSlots + threadIdx.x] = s_trace_[threadIdx.x]; \
  } while (0)
// For kernels whose threads do not all meet at the end: thread `thr` writes its stamp k straight
// to the store (the same layout), the first time it passes it.
#define DSA_STAMP_DIRECT(store, k, thr)                                                     \
  do {                                                                                      \
    if (threadIdx.x == (thr) && s_trace_[k] == 0ull && blockIdx.x < ::dsa::kTraceCtas) {    \
      s_trace_[k] = 1ull;                                                                   \
      (store)[blockIdx.x * 2 * ::dsa::kTraceSlots + (k)] = clock64();                       \
      (store)[blockIdx.x * 2 * ::dsa::kTraceSlots + ::dsa::kTraceSlots + (k)] =             \
          ::dsa::global_timer_ns();                                                         \
    }                                                                                       \
  } while (0)
#else
#define DSA_STAMP_DIRECT(store, k, thr) \
  do {                                  \
  } while (0)
#define DSA_TRACE_BEGIN() \
  do {                    \
  } while (0)
#define DSA_STAMP(k) \
  do {               \
  } while (0)
#define DSA_TRACE_END(store) \
  do {                       \
  } while (0)
#endif

}  // namespace dsa
