// Persistent split-K sparse attention over many rows: one launch, one CTA per SM.
//
// Work partition (stream-K over page slots): every dense (request, KV head) row owns idx_stride
// consecutive slots of one global slot space; CTA c of the n active CTAs takes the slots
// [floor(c T / n), floor((c + 1) T / n)) of the T slots, so every CTA streams the same number of
// selected pages whatever the number of rows.  The slots of one row inside one CTA form a unit.
// A row that lies inside one CTA is finished by that CTA directly; a row cut across CTAs leaves
// one partial record per CTA (at most two per CTA: its first and its last row), and the CTA that
// takes the row's last ticket merges them in CTA order.  No CTA ever waits for another.
//
// Inside a CTA, warp 8 is a TMA producer: it sets up the barriers alone and, before its general
// loop, issues the first unit's first pages from a short straight-line path; the loop then
// resolves 32 page-table entries at a time and streams whole pages through a ring (bf16: two 3-D
// tensor loads per page into about 128 KB; quantised blocks: one bulk copy each, up to 64 stages
// in 160 KB), several lanes issuing at once.  Warps 0..7 attend with the mma core.  Every (stage,
// 16-token tile) slot of the ring belongs to one consumer warp for the whole launch, so a warp
// waits only for the pages it computes on, it waits on every phase of its stages in order (a
// phase-parity wait is only unambiguous for a waiter that never skips a phase), and each stage is
// released by exactly the warps that read it.  The producer also publishes each unit (its row,
// selected slots and request length, and the row's G query vectors by a 1-D bulk copy) through a
// two-slot mailbox, so the consumers never touch global memory before their epilogues.
// The page format (bf16, KV8, KV4) is a template parameter, and so is the tile orientation of the
// quantised formats (transposed for query groups of at most 8).
#include "attn_core.cuh"
#include <cuda_fp8.h>

#include <type_traits>

#include "internal.h"

namespace dsa {
#ifdef DSA_TIMELINE
__device__ unsigned long long g_trace_stream[kTraceCtas * 2 * kTraceSlots];
#endif
namespace {

constexpr int kSW = 8;                     // consumer warps
constexpr int kSThreads = (kSW + 1) * 32;  // + one TMA producer warp
constexpr int kSConsumers = kSW * 32;
constexpr int kSMaxHeads = 1024;           // KV heads the dense-head table can hold
constexpr int kUnitPadTokens = 128;        // empty slots per dense row, in tokens of pages
constexpr int kIssueLanes = 4;             // producer lanes issuing page loads at once
constexpr int kMiscWords = 32 + 2 * kStreamMaxStages;  // shared words before the head tables

struct SLayout {
  uint32_t stage_stride, merge_off, q_off, bar_off, misc_off, total;
};

// merge area: per warp G rows of O (fp32) and G (m, l) pairs; later the row merge's weights.
// q: two unpadded [16][128] bf16 query tiles (mailbox slots).  bars: [S] full, [S] empty, then the
// mailbox's [2] full and [2] empty.
// kv8: a stage holds a KV8 page block (e4m3 K rows, V rows, then the two fp32 scale rows); the
// consumers read the codes straight into tensor-core operands (no decoded copy in shared memory).
// Page formats of the stream: bf16 pools (tensor-map loads) or quantised blocks (one bulk copy per
// page block): KV8 (264 bytes per token) and KV4 (136 bytes per token).
enum : int { kFmtBf16 = 0, kFmtKv8 = 8, kFmtKv4 = 4 };
__host__ __device__ constexpr uint32_t block_bytes_per_token(int fmt) {
  return fmt == kFmtKv8 ? 264u : fmt == kFmtKv4 ? 136u : 512u;
}

__host__ __device__ inline SLayout slayout(int page, int stages, int G, int fmt = kFmtBf16) {
  SLayout L;
  // (a quantised block arrives by a 1-D bulk copy: 16-byte alignment is all it needs; the bf16
  // pages' 128-byte-swizzled tensor loads want 1024)
  L.stage_stride = fmt == kFmtBf16 ? 512u * page
                                   : (block_bytes_per_token(fmt) * page + 15u) & ~15u;
  L.merge_off = ((L.stage_stride * stages) + 1023u) & ~1023u;
  L.q_off = L.merge_off + static_cast<uint32_t>(kSW * G * (kHeadDim + 2) * 4 + 127) / 128 * 128;
  L.bar_off = L.q_off + 2u * 16u * kHeadDim * 2u;
  L.misc_off = L.bar_off + 16u * static_cast<uint32_t>(stages) + 32u;
  L.total = ((L.misc_off + 4u * kMiscWords + 8u * kSMaxHeads + 1023u) & ~1023u) + 1024u;
  return L;
}

// ---- KV8 tiles, read from the codes in registers.  Products run in f16 (an e4m3 value is exact
// in f16): S = Q . codes_K^T, then each token's logit times its K scale; P times each token's V
// scale, then O += (P * s_V) . codes_V.  A code row keeps its 16-byte pieces XOR-permuted by the
// row's index mod 8 (the KV8 layout), so the loads below hit distinct banks.

// Two e4m3 values (the low 16 bits of w) as an f16 pair.
DSA_DEV uint32_t e4m3x2_f16x2(uint32_t w) {
  const __half2_raw h =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

DSA_DEV uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

DSA_DEV void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Query fragments (f16) for the KV8 scores.  The head dims are permuted inside the k-steps so that
// a lane's K operand is one 32-byte run of a code row: lane column tig owns dims 32 tig .. +31,
// k-step ks takes dims 32 tig + 4 ks .. +3 of them (+0, +1 as k = 2 tig, 2 tig + 1; +2, +3 as
// k = 2 tig + 8, + 9).  sQ: 16 rows of 128 bf16.
DSA_DEV void load_q_frags_kv8(const __nv_bfloat16* sQ, uint32_t (&qa)[8][4]) {
  const int lane = threadIdx.x & 31;
  const int r0 = lane >> 2, tig = lane & 3;
  auto f16_pair = [](uint32_t bf2) {
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&bf2);
    const float2 f = __bfloat1622float2(b);
    return pack_f16(f.x, f.y);
  };
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c = 32 * tig + 4 * ks;
    const uint2 lo = *reinterpret_cast<const uint2*>(sQ + r0 * kHeadDim + c);
    const uint2 hi = *reinterpret_cast<const uint2*>(sQ + (r0 + 8) * kHeadDim + c);
    qa[ks][0] = f16_pair(lo.x);
    qa[ks][1] = f16_pair(hi.x);
    qa[ks][2] = f16_pair(lo.y);
    qa[ks][3] = f16_pair(hi.y);
  }
}

// S = Q . codes^T for the 16 code rows at kc (rows 16t .. 16t + 15 of a page block).
DSA_DEV void tile_scores_kv8(const uint32_t (&qa)[8][4], const uint8_t* kc, float (&sc)[2][4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  float acc[2][2][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[c][nt][e] = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const uint8_t* row = kc + (nt * 8 + g) * 128;  // token nt * 8 + g; its index mod 8 is g
    const uint4 w0 = *reinterpret_cast<const uint4*>(row + (((2 * tig) ^ g) << 4));
    const uint4 w1 = *reinterpret_cast<const uint4*>(row + (((2 * tig + 1) ^ g) << 4));
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_f16(acc[ks & 1][nt], qa[ks], e4m3x2_f16x2(w[ks]), e4m3x2_f16x2(w[ks] >> 16));
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[nt][e] = acc[0][nt][e] + acc[1][nt][e];
}

// ---- KV4 tiles.  A code is a nibble u (value u - 8); f16(1024 + u) - 1032 is that value exactly,
// so two nibbles placed in the mantissas of a 0x6400 pair and shifted down by one packed f16
// subtraction give an f16 operand pair.  The same dim permutations as the KV8 tiles; the 64-byte
// code row of token r sits at row r ^ ((r >> 1) & 1) of its tile (r mod 4 is the same in both).

DSA_DEV int kv4_row(int r) { return r ^ ((r >> 1) & 1); }

// f16 pair (lo, hi) = (nibble of `w` at bit `a` - 8, nibble at bit `b` - 8)
DSA_DEV uint32_t kv4_pair(uint32_t w, int a, int b) {
  const uint32_t bits = ((w >> a) & 0xfu) | (((w >> b) & 0xfu) << 16) | 0x64006400u;
  const uint32_t off = 0x64086408u;  // (1032, 1032)
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&bits),
                            *reinterpret_cast<const __half2*>(&off));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The same for the nibbles at bits a and a + 16 of w: one shift and one mask-and-or.
DSA_DEV uint32_t kv4_pair16(uint32_t w, int a) {
  const uint32_t bits = ((w >> a) & 0x000f000fu) | 0x64006400u;
  const uint32_t off = 0x64086408u;
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&bits),
                            *reinterpret_cast<const __half2*>(&off));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// S = Q . codes^T for the 16 code rows at kc (the tile's rows of a KV4 page block).  Lane column
// tig reads dims 32 tig .. +31 of its token: 16 bytes, k-step ks taking the nibbles of dims
// 32 tig + 4 ks .. +3 (one 16-bit half of word ks / 2).
DSA_DEV void tile_scores_kv4(const uint32_t (&qa)[8][4], const uint8_t* kc, float (&sc)[2][4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  float acc[2][2][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[c][nt][e] = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const uint4 w4 = *reinterpret_cast<const uint4*>(kc + kv4_row(nt * 8 + g) * 64 + 16 * tig);
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int h = 16 * (ks & 1);
      mma_f16(acc[ks & 1][nt], qa[ks], kv4_pair(w[ks >> 1], h, h + 4),
              kv4_pair(w[ks >> 1], h + 8, h + 12));
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[nt][e] = acc[0][nt][e] + acc[1][nt][e];
}

// O += (P * s_V) . codes_V for the tile's V code rows at vc (pa: the P fragment, already scaled).
// n-tile j, column c holds dim 16 c + j (the KV8 output permutation): lane g reads dims 16 g ..
// + 15 (8 bytes) of tokens 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9.
DSA_DEV void tile_pv_kv4(WarpSoftmaxState& st, const uint32_t (&pa)[4], const uint8_t* vc) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  uint2 rv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 2 * tig + (i & 1) + (i >> 1) * 8;
    rv[i] = *reinterpret_cast<const uint2*>(vc + kv4_row(r) * 64 + 8 * g);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {  // dims 16 g + 8 half .. + 7
    const uint32_t w0 = half ? rv[0].y : rv[0].x, w1 = half ? rv[1].y : rv[1].x;
    const uint32_t w2 = half ? rv[2].y : rv[2].x, w3 = half ? rv[3].y : rv[3].x;
#pragma unroll
    for (int quad = 0; quad < 2; ++quad) {  // dims + 4 quad .. + 3: bytes 2 quad, 2 quad + 1
      // rows (2 tig, 2 tig + 1) and (2 tig + 8, 2 tig + 9) side by side, 16 bits each
      const uint32_t sel = quad ? 0x7632u : 0x5410u;
      const uint32_t x01 = __byte_perm(w0, w1, sel), x23 = __byte_perm(w2, w3, sel);
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int j = 8 * half + 4 * quad + n;
        mma_f16(st.o[j], pa, kv4_pair16(x01, 4 * n), kv4_pair16(x23, 4 * n));
      }
    }
  }
}

// Online-softmax update with the tile's logits (q . codes in sc; ks / vs: the 16 tokens' K and V
// scales), then O += (P * s_V) . codes_V over KV8 (FMT 8) or KV4 (FMT 4) code rows at vc.  The
// output dims are permuted: n-tile j, column c holds dim 16 c + j, so that a lane's V operand is
// one piece of each of its four code rows (16 bytes of KV8, 8 bytes of KV4).
template <int FMT>
DSA_DEV void tile_softmax_pv_q(WarpSoftmaxState& st, float (&sc)[2][4], float scale_log2,
                               uint32_t valid, const uint8_t* vc, const float* ks,
                               const float* vs) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const float2 k0 = *reinterpret_cast<const float2*>(ks + 2 * tig);
  const float2 k1 = *reinterpret_cast<const float2*>(ks + 8 + 2 * tig);
  const float kscale[2][2] = {{k0.x, k0.y}, {k1.x, k1.y}};
  float x[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = nt * 8 + tig * 2 + (e & 1);
      x[nt][e] = ((valid >> col) & 1u) ? sc[nt][e] * kscale[nt][e & 1] * scale_log2 : -INFINITY;
    }
  float mx[2];
  mx[0] = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
  mx[1] = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
  }
  float alpha[2], mnew[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mnew[r] = fmaxf(st.m[r], mx[r]);
    alpha[r] = (mnew[r] == -INFINITY) ? 1.f : fast_exp2(st.m[r] - mnew[r]);
  }
  float p[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = e >> 1;
      p[nt][e] = (mnew[r] == -INFINITY) ? 0.f : fast_exp2(x[nt][e] - mnew[r]);
    }
  st.l[0] = st.l[0] * alpha[0] + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
  st.l[1] = st.l[1] * alpha[1] + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
  st.m[0] = mnew[0];
  st.m[1] = mnew[1];
  if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      st.o[j][0] *= alpha[0];
      st.o[j][1] *= alpha[0];
      st.o[j][2] *= alpha[1];
      st.o[j][3] *= alpha[1];
    }
  }
  // P * s_V (0 for tokens that take no part, whatever their scale holds)
  const float2 v0 = *reinterpret_cast<const float2*>(vs + 2 * tig);
  const float2 v1 = *reinterpret_cast<const float2*>(vs + 8 + 2 * tig);
  const float vscale[2][2] = {{v0.x, v0.y}, {v1.x, v1.y}};
  float pv[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = nt * 8 + tig * 2 + (e & 1);
      pv[nt][e] = ((valid >> col) & 1u) ? p[nt][e] * vscale[nt][e & 1] : 0.f;
    }
  uint32_t pa[4];
  pa[0] = pack_f16(pv[0][0], pv[0][1]);
  pa[1] = pack_f16(pv[0][2], pv[0][3]);
  pa[2] = pack_f16(pv[1][0], pv[1][1]);
  pa[3] = pack_f16(pv[1][2], pv[1][3]);
  if constexpr (FMT == 4) {  // (a nibble always decodes to a finite value: nothing to clear)
    tile_pv_kv4(st, pa, vc);
  } else {
    // V operand of n-tile j: tokens 2 tig, 2 tig + 1 (b0) and 2 tig + 8, + 9 (b1) at dim 16 g + j:
    // byte j of the 16-byte piece g of those four code rows (zeros for tokens that take no part,
    // so that stale codes never meet a zero probability)
    uint4 rv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 2 * tig + (i & 1) + (i >> 1) * 8;
      rv[i] = *reinterpret_cast<const uint4*>(vc + r * 128 + ((g ^ (r & 7)) << 4));
      if (!((valid >> r) & 1u)) rv[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    const uint32_t* w0 = reinterpret_cast<const uint32_t*>(&rv[0]);
    const uint32_t* w1 = reinterpret_cast<const uint32_t*>(&rv[1]);
    const uint32_t* w2 = reinterpret_cast<const uint32_t*>(&rv[2]);
    const uint32_t* w3 = reinterpret_cast<const uint32_t*>(&rv[3]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // dims 16 g + 4 q .. + 3
      const uint32_t a01 = __byte_perm(w0[q], w1[q], 0x5140), b01 = __byte_perm(w0[q], w1[q], 0x7362);
      const uint32_t a23 = __byte_perm(w2[q], w3[q], 0x5140), b23 = __byte_perm(w2[q], w3[q], 0x7362);
      mma_f16(st.o[4 * q], pa, e4m3x2_f16x2(a01), e4m3x2_f16x2(a23));
      mma_f16(st.o[4 * q + 1], pa, e4m3x2_f16x2(a01 >> 16), e4m3x2_f16x2(a23 >> 16));
      mma_f16(st.o[4 * q + 2], pa, e4m3x2_f16x2(b01), e4m3x2_f16x2(b23));
      mma_f16(st.o[4 * q + 3], pa, e4m3x2_f16x2(b01 >> 16), e4m3x2_f16x2(b23 >> 16));
    }
  }
}

// ---- Transposed tiles (quantised pages, query groups of at most 8).  S^T = codes_K . Q^T puts
// the tile's 16 tokens on the m16 rows of the tensor-core product and the group on n8, so each
// product is one mma per k-step (the untransposed tiles spend two, three quarters of their rows
// empty at G = 4).  The probabilities leave the scores' accumulator layout as the next product's
// B operand through two in-register 8x8 transposes (movmatrix).  O^T = codes_V^T . (P * s_V)^T
// takes 8 m16 tiles of head dims: m-tile mt, row r < 8 is dim 16 r + 2 mt and row r + 8 is dim
// 16 r + 2 mt + 1, so that a lane's V operands are the same pieces of four code rows as in the
// untransposed tiles, and each lane ends holding adjacent dims of its two query heads.

struct WarpStateT {
  float o[8][4];  // O^T m-tile mt: rows g, g + 8 (dims 16 g + 2 mt, + 1), columns 2 tig, 2 tig + 1
  float m[2];     // running max (log2 units) of query heads 2 tig, 2 tig + 1
  float l[2];     // this lane's partial denominators of the same heads
};

DSA_DEV void state_init(WarpStateT& st) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[j][e] = 0.f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
}

// The denominators summed over the eight lanes (g) that hold a head's tokens.
DSA_DEV void state_finish(WarpStateT& st) {
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], o);
}

DSA_DEV uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// B fragments of Q^T (f16): qb[ks][0] = head g's dims d, d + 1 and qb[ks][1] its dims d + 2, d + 3,
// d = 32 tig + 4 ks (the K operand's dim permutation); heads g >= G read the zero rows of sQ.
DSA_DEV void load_qT_frags(const __nv_bfloat16* sQ, uint32_t (&qb)[8][4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  auto f16_pair = [](uint32_t bf2) {
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&bf2);
    const float2 f = __bfloat1622float2(b);
    return pack_f16(f.x, f.y);
  };
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint2 v = *reinterpret_cast<const uint2*>(sQ + g * kHeadDim + 32 * tig + 4 * ks);
    qb[ks][0] = f16_pair(v.x);
    qb[ks][1] = f16_pair(v.y);
  }
}

// The same for the KV4 transposed scores: k-step ks = 2 i + s takes dims 32 tig + 8 i + 2 s,
// + 2 s + 4 (qb[ks][0]) and + 2 s + 1, + 2 s + 5 (qb[ks][1]).
DSA_DEV void load_qT_frags_kv4(const __nv_bfloat16* sQ, uint32_t (&qb)[8][4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const __nv_bfloat16* row = sQ + g * kHeadDim + 32 * tig;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int d = 8 * (ks >> 1) + 2 * (ks & 1);
    qb[ks][0] = pack_f16(__bfloat162float(row[d]), __bfloat162float(row[d + 4]));
    qb[ks][1] = pack_f16(__bfloat162float(row[d + 1]), __bfloat162float(row[d + 5]));
  }
}

// S^T for the tile's 16 code rows at kc: sc[0], sc[1] = token g, heads 2 tig, 2 tig + 1;
// sc[2], sc[3] = token g + 8, the same heads.
template <int FMT>
DSA_DEV void tileT_scores(const uint32_t (&qb)[8][4], const uint8_t* kc, float (&sc)[4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  float acc[2][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[c][e] = 0.f;
  if constexpr (FMT == 8) {
    // rows g and g + 8 (both at index g mod 8): the 16-byte pieces of dims 32 tig .. + 31
    const uint8_t* ra = kc + g * 128;
    const uint8_t* rb = kc + (g + 8) * 128;
    const uint4 a0 = *reinterpret_cast<const uint4*>(ra + (((2 * tig) ^ g) << 4));
    const uint4 a1 = *reinterpret_cast<const uint4*>(ra + (((2 * tig + 1) ^ g) << 4));
    const uint4 b0 = *reinterpret_cast<const uint4*>(rb + (((2 * tig) ^ g) << 4));
    const uint4 b1 = *reinterpret_cast<const uint4*>(rb + (((2 * tig + 1) ^ g) << 4));
    const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t af[4] = {e4m3x2_f16x2(wa[ks]), e4m3x2_f16x2(wb[ks]),
                              e4m3x2_f16x2(wa[ks] >> 16), e4m3x2_f16x2(wb[ks] >> 16)};
      mma_f16(acc[ks & 1], af, qb[ks][0], qb[ks][1]);
    }
  } else {
    // k-step ks = 2 i + s of lane tig: word i of its 16 bytes (dims 32 tig + 8 i .. + 7), the
    // dims at nibbles 2 s, 2 s + 4 (k = 2 tig, 2 tig + 1) and 2 s + 1, 2 s + 5 (k = 2 tig + 8, + 9):
    // each pair 16 bits apart (the query fragments take the same dims, load_qT_frags_kv4)
    const uint4 a4 = *reinterpret_cast<const uint4*>(kc + kv4_row(g) * 64 + 16 * tig);
    const uint4 b4 = *reinterpret_cast<const uint4*>(kc + kv4_row(g + 8) * 64 + 16 * tig);
    const uint32_t wa[4] = {a4.x, a4.y, a4.z, a4.w};
    const uint32_t wb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int sh = 8 * (ks & 1);
      const uint32_t af[4] = {kv4_pair16(wa[ks >> 1], sh), kv4_pair16(wb[ks >> 1], sh),
                              kv4_pair16(wa[ks >> 1], sh + 4), kv4_pair16(wb[ks >> 1], sh + 4)};
      mma_f16(acc[ks & 1], af, qb[ks][0], qb[ks][1]);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) sc[e] = acc[0][e] + acc[1][e];
}

// Online-softmax update of the transposed tile (logits q . codes in sc, ks / vs: the 16 tokens'
// K and V scales), then O^T += codes_V^T . (P * s_V)^T over the tile's V code rows at vc.
template <int FMT>
DSA_DEV void tileT_softmax_pv(WarpStateT& st, const float (&sc)[4], float scale_log2,
                              uint32_t valid, const uint8_t* vc, const float* ks,
                              const float* vs) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const bool va = (valid >> g) & 1u, vb = (valid >> (g + 8)) & 1u;
  const float ka = ks[g] * scale_log2, kb = ks[g + 8] * scale_log2;
  float x[4];
  x[0] = va ? sc[0] * ka : -INFINITY;
  x[1] = va ? sc[1] * ka : -INFINITY;
  x[2] = vb ? sc[2] * kb : -INFINITY;
  x[3] = vb ? sc[3] * kb : -INFINITY;
  float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], o));
  float alpha[2], mnew[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mnew[r] = fmaxf(st.m[r], mx[r]);
    alpha[r] = (mnew[r] == -INFINITY) ? 1.f : fast_exp2(st.m[r] - mnew[r]);
  }
  float p[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int r = e & 1;
    p[e] = (mnew[r] == -INFINITY) ? 0.f : fast_exp2(x[e] - mnew[r]);
  }
  st.l[0] = st.l[0] * alpha[0] + (p[0] + p[2]);
  st.l[1] = st.l[1] * alpha[1] + (p[1] + p[3]);
  st.m[0] = mnew[0];
  st.m[1] = mnew[1];
  if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      st.o[j][0] *= alpha[0];
      st.o[j][1] *= alpha[1];
      st.o[j][2] *= alpha[0];
      st.o[j][3] *= alpha[1];
    }
  }
  // P * s_V (0 for tokens that take no part, whatever their scale holds), then the B operand:
  // tokens 2 tig, 2 tig + 1 (b0) and 2 tig + 8, + 9 (b1) of head g
  const float sa = va ? vs[g] : 0.f, sb = vb ? vs[g + 8] : 0.f;
  const uint32_t b0 = movmatrix_trans(pack_f16(p[0] * sa, p[1] * sa));
  const uint32_t b1 = movmatrix_trans(pack_f16(p[2] * sb, p[3] * sb));
  if constexpr (FMT == 8) {
    // the 16-byte pieces g (dims 16 g .. + 15) of code rows 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9
    // (zeros for tokens that take no part, so that stale codes never meet a zero probability)
    uint4 rv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 2 * tig + (i & 1) + (i >> 1) * 8;
      rv[i] = *reinterpret_cast<const uint4*>(vc + r * 128 + ((g ^ (r & 7)) << 4));
      if (!((valid >> r) & 1u)) rv[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    const uint32_t* w0 = reinterpret_cast<const uint32_t*>(&rv[0]);
    const uint32_t* w1 = reinterpret_cast<const uint32_t*>(&rv[1]);
    const uint32_t* w2 = reinterpret_cast<const uint32_t*>(&rv[2]);
    const uint32_t* w3 = reinterpret_cast<const uint32_t*>(&rv[3]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // dims 16 g + 4 q .. + 3: m-tiles 2 q and 2 q + 1
      const uint32_t a01 = __byte_perm(w0[q], w1[q], 0x5140), c01 = __byte_perm(w0[q], w1[q], 0x7362);
      const uint32_t a23 = __byte_perm(w2[q], w3[q], 0x5140), c23 = __byte_perm(w2[q], w3[q], 0x7362);
      const uint32_t fa[4] = {e4m3x2_f16x2(a01), e4m3x2_f16x2(a01 >> 16), e4m3x2_f16x2(a23),
                              e4m3x2_f16x2(a23 >> 16)};
      const uint32_t fc[4] = {e4m3x2_f16x2(c01), e4m3x2_f16x2(c01 >> 16), e4m3x2_f16x2(c23),
                              e4m3x2_f16x2(c23 >> 16)};
      mma_f16(st.o[2 * q], fa, b0, b1);
      mma_f16(st.o[2 * q + 1], fc, b0, b1);
    }
  } else {
    // 8 bytes (dims 16 g .. + 15) of each of the four code rows; a nibble always decodes to a
    // finite value, so nothing needs clearing
    uint2 rv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 2 * tig + (i & 1) + (i >> 1) * 8;
      rv[i] = *reinterpret_cast<const uint2*>(vc + kv4_row(r) * 64 + 8 * g);
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // dims 16 g + 8 half .. + 7: m-tiles 4 half .. + 3
      const uint32_t w0 = half ? rv[0].y : rv[0].x, w1 = half ? rv[1].y : rv[1].x;
      const uint32_t w2 = half ? rv[2].y : rv[2].x, w3 = half ? rv[3].y : rv[3].x;
#pragma unroll
      for (int quad = 0; quad < 2; ++quad) {  // dims + 4 quad .. + 3: m-tiles 4 half + 2 quad, + 1
        const uint32_t sel = quad ? 0x7632u : 0x5410u;
        const uint32_t x01 = __byte_perm(w0, w1, sel), x23 = __byte_perm(w2, w3, sel);
#pragma unroll
        for (int n = 0; n < 2; ++n) {  // dims + 2 n (rows g) and + 2 n + 1 (rows g + 8)
          const uint32_t fa[4] = {kv4_pair16(x01, 8 * n), kv4_pair16(x01, 8 * n + 4),
                                  kv4_pair16(x23, 8 * n), kv4_pair16(x23, 8 * n + 4)};
          mma_f16(st.o[4 * half + 2 * quad + n], fa, b0, b1);
        }
      }
    }
  }
}

// ---- Transposed tiles over bf16 pages (query groups of at most 8): the K tile is the A operand
// as it lies in the 128-byte-swizzled stage (ldmatrix), the V tile is V^T through a transposing
// ldmatrix, and O^T's m-tile mt holds dims 16 mt .. + 15 in order (rows g and g + 8).

// B fragments of Q^T in natural dim order: qb[ks][0] = head g's dims 16 ks + 2 tig, + 1 and
// qb[ks][1] its dims 16 ks + 2 tig + 8, + 9 (bf16 pairs).
DSA_DEV void load_qT_frags_bf16(const __nv_bfloat16* sQ, uint32_t (&qb)[8][4]) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qb[ks][0] = *reinterpret_cast<const uint32_t*>(sQ + g * kHeadDim + 16 * ks + 2 * tig);
    qb[ks][1] = *reinterpret_cast<const uint32_t*>(sQ + g * kHeadDim + 16 * ks + 2 * tig + 8);
  }
}

// S^T for tokens [row0, row0 + 16) of a staged page (kbase: the K box of dims 0..63; dims 64..127
// follow at + page * 128): sc as in tileT_scores.
DSA_DEV void tileT_scores_bf16(const uint32_t (&qb)[8][4], uint32_t kbase, int page, int row0,
                               float (&sc)[4]) {
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3;
  const uint32_t tok = static_cast<uint32_t>(row0 + (mi & 1) * 8 + (lane & 7));
  const uint32_t half_stride = static_cast<uint32_t>(page * 128);
  float acc[2][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[c][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t chunk = static_cast<uint32_t>(2 * ks + (mi >> 1));
    uint32_t af[4];
    ldsm_x4(kbase + (chunk >> 3) * half_stride + sw128(tok, chunk & 7u), af[0], af[1], af[2],
            af[3]);
    mma_bf16(acc[ks & 1], af, qb[ks][0], qb[ks][1]);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) sc[e] = acc[0][e] + acc[1][e];
}

// Online-softmax update of the transposed bf16 tile, then O^T += V^T . P^T (vbase: the V box of
// dims 0..63 of the staged page).
DSA_DEV void tileT_softmax_pv_bf16(WarpStateT& st, const float (&sc)[4], float scale_log2,
                                   uint32_t valid, uint32_t vbase, int page, int row0) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const bool va = (valid >> g) & 1u, vb = (valid >> (g + 8)) & 1u;
  float x[4];
  x[0] = va ? sc[0] * scale_log2 : -INFINITY;
  x[1] = va ? sc[1] * scale_log2 : -INFINITY;
  x[2] = vb ? sc[2] * scale_log2 : -INFINITY;
  x[3] = vb ? sc[3] * scale_log2 : -INFINITY;
  float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
  for (int r = 0; r < 2; ++r)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], o));
  float alpha[2], mnew[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mnew[r] = fmaxf(st.m[r], mx[r]);
    alpha[r] = (mnew[r] == -INFINITY) ? 1.f : fast_exp2(st.m[r] - mnew[r]);
  }
  float p[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int r = e & 1;
    p[e] = (mnew[r] == -INFINITY) ? 0.f : fast_exp2(x[e] - mnew[r]);
  }
  st.l[0] = st.l[0] * alpha[0] + (p[0] + p[2]);
  st.l[1] = st.l[1] * alpha[1] + (p[1] + p[3]);
  st.m[0] = mnew[0];
  st.m[1] = mnew[1];
  if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      st.o[j][0] *= alpha[0];
      st.o[j][1] *= alpha[1];
      st.o[j][2] *= alpha[0];
      st.o[j][3] *= alpha[1];
    }
  }
  const uint32_t b0 = movmatrix_trans(pack_bf16(p[0], p[1]));
  const uint32_t b1 = movmatrix_trans(pack_bf16(p[2], p[3]));
  const int mi = lane >> 3;
  const uint32_t tok = static_cast<uint32_t>(row0 + (mi >> 1) * 8 + (lane & 7));
  const uint32_t half_stride = static_cast<uint32_t>(page * 128);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {  // dims 16 mt .. + 15
    const uint32_t chunk = static_cast<uint32_t>(2 * mt + (mi & 1));
    uint32_t af[4];
    ldsm_x4_t(vbase + (chunk >> 3) * half_stride + sw128(tok, chunk & 7u), af[0], af[1], af[2],
              af[3]);
    mma_bf16(st.o[mt], af, b0, b1);
  }
}

// Shared position of output dim d of query head r in the KV8 path's merge area: the pieces of 16
// dims are XOR-permuted by the writer's column pair and row, so that the fragment stores of a warp
// spread over the banks.
DSA_DEV int kv8_o_pos(int r, int d) {
  const int c = d >> 4;
  return (d & ~15) | ((d & 15) ^ (((c >> 1) & 3) | ((r & 3) << 2)));
}

// Slot range [beg, end) of the active CTA c among n over T slots.
// (32-bit divisions when the operands fit: a 64-bit division is a long subroutine, and these sit
// on every CTA's start-up path)
__device__ __forceinline__ long long slot_start(long long c, long long T, long long n) {
  const unsigned long long p = static_cast<unsigned long long>(c * T);
  if (p <= 0xffffffffull && static_cast<unsigned long long>(n) <= 0xffffffffull)
    return static_cast<unsigned>(p) / static_cast<unsigned>(n);
  return c * T / n;
}

// x / d for x >= 0, d > 0.
__device__ __forceinline__ long long div_slots(long long x, long long d) {
  if (static_cast<unsigned long long>(x) <= 0xffffffffull &&
      static_cast<unsigned long long>(d) <= 0xffffffffull)
    return static_cast<unsigned>(x) / static_cast<unsigned>(d);
  return x / d;
}

// Index of the active CTA whose slot range holds slot x.
__device__ __forceinline__ int slot_owner(long long x, long long T, long long n) {
  return static_cast<int>(div_slots((x + 1) * n - 1, T));
}

DSA_DEV bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 50000000ull) return false;
  return true;
}

// acq_rel fetch-add at GPU scope: publishes this CTA's records (ordered before it by the CTA
// barrier) and, for the last arrival, makes the other CTAs' records visible.
DSA_DEV int ticket_add(int32_t* p) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

// STREAMING: the launch also serves the streaming heads (a second region of the slot space);
// without it every streaming-specific path compiles away.
// TR: the transposed tiles (quantised pages, G <= 8).
template <bool STREAMING, int FMT, bool TR = false>
__global__ void __launch_bounds__(kSThreads, 1)
    stream_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const StreamAttnArgs a) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  const KvView& kv = a.kv;
  const int page = kv.p;
  const int S = a.stages;
  const int G = kv.G;
  const int tiles = page / 16;
  constexpr bool KV8 = FMT == kFmtKv8, KV4 = FMT == kFmtKv4, QNT = KV8 || KV4;
  constexpr uint32_t kBpt = block_bytes_per_token(FMT);  // bytes a page brings per token
  const SLayout lay = slayout(page, S, G, FMT);
  float* sO = reinterpret_cast<float*>(smem + lay.merge_off);  // [kSW][G][128]
  float* sM = sO + kSW * G * kHeadDim;                          // [kSW][G]
  float* sL = sM + kSW * G;                                     // [kSW][G]
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + lay.q_off);  // [2][16][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  uint64_t* qbars = bars + 2 * S;  // mailbox: [2] full, [2] empty
  int* misc = reinterpret_cast<int*>(smem + lay.misc_off);
  volatile int* abort_flag = misc;          // [0]
  volatile int* last_flag = misc + 1;       // [1], [2]: ticket outcomes of the cut rows
  volatile int* issued = misc + 3;          // [3] ring positions the producer has issued
  volatile int* producer_done = misc + 4;   // [4]
  int* n_dense_heads = misc + 5;            // [5]
  int* n_stream_heads = misc + 6;           // [6]
  int* desc = misc + 8;                     // [8, 16): mailbox [2][row, beg, end, len]
  int* desc_kind = misc + 16;               // [16, 18): mailbox [2]: 1 for a streaming unit
  // [20, 28): the cut rows' geometry (see cut_info below)
  volatile int* stage_ok = misc + 32;       // [32, 32 + S): did the producer load this stage
  volatile int* stage_pos = misc + 32 + kStreamMaxStages;  // [.., + S): its page position
  int* dense_heads = misc + kMiscWords;     // [kMiscWords, + Hkv)
  int* stream_heads = misc + kMiscWords + kSMaxHeads;  // [.., + Hkv) when streaming units are on
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t stage_bytes = lay.stage_stride;           // stage s at smem + s * stage_bytes
  const uint32_t stage_tx = kBpt * page;  // bytes a stage's loads bring
  const uint32_t smem_base = smem_u32(smem);
#ifdef DSA_TIMELINE
  __shared__ unsigned long long s_trace_[2 * kTraceSlots];
  if (tid < 2 * kTraceSlots) s_trace_[tid] = 0ull;
#endif
  DSA_STAMP_DIRECT(g_trace_stream, 0, 0);

  // Set-up.  The producer warp initialises the barriers and the shared words and builds the head
  // lists, then arrives at named barrier 2 without waiting: everything its own start-up path needs
  // it wrote itself, so its first loads go out at once.  The consumers wait at that barrier.
  if (warp == kSW) {
    // one barrier per lane: [S] full, [S] empty (one arrival per 16-token tile of the page), then
    // the mailbox's [2] full and [2] empty
    for (int k = lane; k < 2 * S + 4; k += 32)
      mbar_init(smem_u32(&bars[k]), k < S ? 1 : k < 2 * S ? tiles : k < 2 * S + 2 ? 1 : kSW);
    fence_mbar_init();
    if (lane == 0) {
      misc[0] = 0;
      misc[3] = 0;
      misc[4] = 0;
      if (!QNT) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
      }
    }
    // dense (non-streaming) KV heads in ascending order, 32 heads per ballot; the streaming
    // ones too when this launch serves them
    int nd = 0, ns = 0;
    if (kv.streaming == nullptr) {
      nd = kv.Hkv;
      for (int hh = lane; hh < kv.Hkv; hh += 32) dense_heads[hh] = hh;
    } else {
      for (int h0 = 0; h0 < kv.Hkv; h0 += 32) {
        const int hh = h0 + lane;
        const bool dense = hh < kv.Hkv && kv.streaming[hh] == 0;
        const bool strm = STREAMING && hh < kv.Hkv && !dense;
        const unsigned bal = __ballot_sync(0xffffffffu, dense);
        const unsigned bas = __ballot_sync(0xffffffffu, strm);
        if (dense) dense_heads[nd + __popc(bal & ((1u << lane) - 1u))] = hh;
        if (strm) stream_heads[ns + __popc(bas & ((1u << lane) - 1u))] = hh;
        nd += __popc(bal);
        ns += __popc(bas);
      }
    }
    if (lane == 0) {
      *n_dense_heads = nd;
      *n_stream_heads = ns;
    }
    __syncwarp();
    named_barrier_arrive(2, kSThreads);
    DSA_STAMP_DIRECT(g_trace_stream, 19, kSW * 32);  // producer: set-up done
  } else {
    // query rows G..15 of both mailbox tiles stay zero (the bulk copies write rows < G only)
    for (int e = tid; e < 2 * 16 * 16; e += kSConsumers) {
      const int r = (e >> 4) & 15;
      if (r >= G) reinterpret_cast<uint4*>(sQ)[e] = make_uint4(0, 0, 0, 0);
    }
    named_barrier(2, kSThreads);
  }
  DSA_STAMP_DIRECT(g_trace_stream, 1, 0);  // set-up done (barrier)
  const int nd_heads = *n_dense_heads;
  const int ns_heads = STREAMING ? *n_stream_heads : 0;
  // The slot space: every dense row's idx_stride selection slots followed by `pad` empty slots,
  // then (when streaming heads are served) every streaming row's stream_stride slots, one per page
  // of its sink and local tokens.  A unit is one row's slots; units are numbered dense rows first.
  // The empty slots (about 128 tokens' worth of pages) charge each row boundary for the unit
  // epilogue it costs: a CTA holding two units gets that many fewer pages, instead of finishing
  // one epilogue later than the CTAs holding one.
  const int istride = a.idx_stride;  // selection slots per dense row (the idx row stride)
  const int pad = max(1, kUnitPadTokens / page);
  const int stride = istride + pad, sstride = a.stream_stride;
  const int Nd = kv.B * nd_heads;
  const long long Td = static_cast<long long>(Nd) * stride;
  const long long T = Td + static_cast<long long>(kv.B) * ns_heads * sstride;
  auto unit_of = [&](long long x) -> int {  // the unit holding slot x
    if (!STREAMING || x < Td) return static_cast<int>(div_slots(x, stride));
    return Nd + static_cast<int>(div_slots(x - Td, sstride));
  };
  auto unit_start = [&](int di) -> long long {  // its first slot
    if (!STREAMING || di < Nd) return static_cast<long long>(di) * stride;
    return Td + static_cast<long long>(di - Nd) * sstride;
  };
  auto unit_stride = [&](int di) { return !STREAMING || di < Nd ? stride : sstride; };
  auto unit_row = [&](int di) -> int {  // its (request, KV head) row
    if constexpr (STREAMING) {
      if (di >= Nd) {
        const int e = di - Nd;
        return (e / ns_heads) * kv.Hkv + stream_heads[e % ns_heads];
      }
    }
    if (nd_heads == kv.Hkv) return di;  // every head is a dense one
    return (di / nd_heads) * kv.Hkv + dense_heads[di % nd_heads];
  };
  // a streaming row of length L attends the pages of its sink tokens [0, min(sink, L)), then
  // those of its local tokens [max(0, L - local), L): sink_n pages from position 0, the rest
  // from position first2 (the two runs merge when they touch)
  auto stream_geom = [&](int L, int* sink_n, int* first2) -> int {
    const int npos = (L + page - 1) / page;
    const int sn = (min(a.sink, L) + page - 1) / page;
    const int f2 = max(max(0, L - a.local) / page, sn);
    *sink_n = sn;
    *first2 = f2;
    return sn + max(0, npos - f2);
  };
  // active CTAs: at most one per slot, so that every active CTA holds at least one slot
  const long long n_act = T < static_cast<long long>(gridDim.x) ? T : gridDim.x;
  if (static_cast<long long>(blockIdx.x) >= n_act) return;
  const long long my_beg = slot_start(blockIdx.x, T, n_act);
  const long long my_end = slot_start(blockIdx.x + 1, T, n_act);
  const int d_first = unit_of(my_beg);
  const int n_units = unit_of(my_end - 1) - d_first + 1;

  if (warp == kSW) {
    // ---- producer.  Unit u of this CTA is dense row d_first + u; lane l holds the descriptor of
    // unit ub + l of the current batch of 32.  Chunks of up to 32 selected slots of one unit are
    // software-pipelined: while chunk A's pages are issued, the page-table entries of chunk B and
    // the selections of chunk C are already in flight.
    DSA_STAMP_DIRECT(g_trace_stream, 13, kSW * 32 + (n_units == -12345));
    // a group of NL pages uses NL distinct stages; a quantised page is a single copy, so a group
    // issues more of them (their pages are small: the ring turns over faster)
    const int NL = min(QNT ? 4 * kIssueLanes : kIssueLanes, S);
    int i = 0;                           // ring position
    bool stopped = false;
    // First pages, straight-line.  The general loop below is long code that every CTA runs cold at
    // this point; before entering it, the first unit (when it is a dense one) is published and the
    // first min(S, 16) pages of its slots are issued, from a short path whose loads (count, length,
    // selections; then page-table entries) go out together.  The loop then resumes after them.
    int f_beg = -1;  // the first unit's first slot not yet issued (-1: the short path did not run)
    if (!STREAMING || d_first < Nd) {
      const int row0 = unit_row(d_first);
      const long long r0 = unit_start(d_first);
      const int pb = static_cast<int>(my_beg - r0);
      const int pe = static_cast<int>((my_end < r0 + stride ? my_end : r0 + stride) - r0);
      const int b0 = row0 / kv.Hkv, h0 = row0 - b0 * kv.Hkv;
      const int j = pb + lane;
      const int selv = j < istride ? a.idx[static_cast<size_t>(row0) * istride + j] : -1;
      const int cnt = min(max(a.count[row0], 0), istride);
      const int len = request_len(kv, b0);
      const int beg = min(pb, cnt), end = min(pe, cnt);  // beg == pb whenever beg < end
      if (lane == 0) {  // mailbox slot 0 is free at the start
        desc[0] = row0;
        desc[1] = beg;
        desc[2] = end;
        desc[3] = len;
        desc_kind[0] = 0;
        const uint32_t full = smem_u32(&qbars[0]);
        mbar_arrive_expect_tx(full, static_cast<uint32_t>(G) * kHeadDim * 2);
        bulk_load(smem_u32(sQ),
                  a.q + (static_cast<size_t>(b0) * kv.Hq + static_cast<size_t>(h0) * G) * kHeadDim,
                  static_cast<uint32_t>(G) * kHeadDim * 2, full);
      }
      // ring positions 0..F-1 need no waits: up to 32 quantised pages (a lane each), 16 bf16 ones
      // (two lanes each)
      const int F = max(0, min(min(end - beg, S), QNT ? 32 : 16));
      const int pos = lane < F ? selv : -1;
      const bool in = lane < F && pos >= 0 && pos < (len + page - 1) / page;
      const int raw = in ? kv.page_table[static_cast<size_t>(b0) * kv.max_pages + pos] : -1;
      const bool ok = in && raw >= 0 && raw < kv.num_phys;
      if (in && !ok) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
      DSA_STAMP_DIRECT(g_trace_stream, 12, kSW * 32 + (raw == -12345));
      if constexpr (QNT) {  // lane q issues page q's block: one bulk copy
        if (lane < F) {
          const uint32_t full = smem_u32(&bars[lane]);
          stage_pos[lane] = pos;
          stage_ok[lane] = ok ? 1 : 0;  // both published by the arrive below
          if (!ok) {
            mbar_arrive(full);  // nothing to load: complete the phase with a plain arrival
          } else {
            mbar_arrive_expect_tx(full, stage_tx);
            bulk_load(smem_base + lane * stage_bytes,
                      a.qkv + static_cast<size_t>((raw * kv.Hkv + h0) * page) * kBpt, kBpt * page,
                      full);
          }
        }
      } else {
        // lane 2q (K) and lane 2q + 1 (V) take page q, so that the copies go out page by page
        const int q = lane >> 1;
        const int pos_q = __shfl_sync(0xffffffffu, pos, q);
        const int raw_q = __shfl_sync(0xffffffffu, raw, q);
        const bool ok_q = __shfl_sync(0xffffffffu, ok ? 1 : 0, q) != 0;
        if (q < F) {
          const uint32_t full = smem_u32(&bars[q]);
          const uint32_t dst = smem_base + q * stage_bytes;
          const int rowk = (raw_q * kv.Hkv + h0) * page;
          if ((lane & 1) == 0) {
            stage_pos[q] = pos_q;
            stage_ok[q] = ok_q ? 1 : 0;  // both published by the arrive below
            if (!ok_q)
              mbar_arrive(full);  // nothing to load: complete the phase with a plain arrival
            else
              mbar_arrive_expect_tx(full, stage_tx);
          }
          __syncwarp(0xffffffffu >> (32 - 2 * F));  // the byte count is posted before any copy
          if (ok_q) {
            if ((lane & 1) == 0)
              tma_load_page(dst, &tmK, rowk, full);
            else
              tma_load_page(dst + 2 * page * 128, &tmV, rowk, full);
          }
        }
      }
      if (lane == 0) *issued = F;
      DSA_STAMP_DIRECT(g_trace_stream, 8, kSW * 32);  // producer: its first loads issued
      i = F;
      f_beg = beg + F;
    }
    for (int ub = 0; ub < n_units && !stopped; ub += 32) {
      int t_row = 0, t_beg = 0, t_end = 0, t_len = 0, t_kind = 0;
      {
        const int u = ub + lane;
        if (u < n_units) {
          const int di = d_first + u;
          t_row = unit_row(di);
          const long long r0 = unit_start(di);
          const int us = unit_stride(di);
          const int pb = static_cast<int>((my_beg > r0 ? my_beg : r0) - r0);
          const int pe = static_cast<int>((my_end < r0 + us ? my_end : r0 + us) - r0);
          t_len = request_len(kv, t_row / kv.Hkv);
          t_kind = STREAMING && di >= Nd;
          int sn, f2;
          const int cnt = t_kind ? min(stream_geom(t_len, &sn, &f2), us)
                                 : min(max(a.count[t_row], 0), istride);
          t_beg = min(pb, cnt);
          t_end = min(pe, cnt);
        }
      }
      const int ue = min(n_units, ub + 32);
      DSA_STAMP_DIRECT(g_trace_stream, 10, kSW * 32 + (t_len == -12345) + (t_beg == -12345));
      int uq = ub == 0 && f_beg >= 0 ? 1 : ub;  // next unit to publish (the short path did unit 0)
      // publishes unit u: waits for its mailbox slot, writes the descriptor, copies the queries
      auto publish = [&](int u) -> bool {
        const int slot = u & 1;
        int stop = 0;
        if (lane == 0 && u >= 2 &&
            !mbar_wait(smem_u32(&qbars[2 + slot]), ((u >> 1) - 1) & 1, abort_flag, kv.status))
          stop = 1;
        const int row = __shfl_sync(0xffffffffu, t_row, u - ub);
        const int beg = __shfl_sync(0xffffffffu, t_beg, u - ub);
        const int end = __shfl_sync(0xffffffffu, t_end, u - ub);
        const int len = __shfl_sync(0xffffffffu, t_len, u - ub);
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        const int kind = STREAMING ? __shfl_sync(0xffffffffu, t_kind, u - ub) : 0;
        if (lane == 0) {
          desc[slot * 4 + 0] = row;
          desc[slot * 4 + 1] = beg;
          desc[slot * 4 + 2] = end;
          desc[slot * 4 + 3] = len;
          desc_kind[slot] = kind;
          const uint32_t full = smem_u32(&qbars[slot]);
          const int b = row / kv.Hkv, h = row % kv.Hkv;
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(G) * kHeadDim * 2);
          bulk_load(smem_u32(sQ + slot * 16 * kHeadDim),
                    a.q + (static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G) * kHeadDim,
                    static_cast<uint32_t>(G) * kHeadDim * 2, full);
        }
        return true;
      };
      // first chunk at or after slot `base` of unit u (u == ue: none left in this batch)
      auto seek = [&](int u, int base, int* cu, int* cb) {
        while (u < ue) {
          const int e = __shfl_sync(0xffffffffu, t_end, u - ub);
          if (base < e) break;
          ++u;
          if (u < ue) base = __shfl_sync(0xffffffffu, t_beg, u - ub);
        }
        *cu = u;
        *cb = base;
      };
      // lane's selected position in chunk (u, base), -1 past the unit's end
      auto load_sel = [&](int u, int base) -> int {
        if (u >= ue) return -1;
        const int row = __shfl_sync(0xffffffffu, t_row, u - ub);
        const int e = __shfl_sync(0xffffffffu, t_end, u - ub);
        const int j = base + lane;
        if (STREAMING) {  // every lane takes the shuffles, before any lane returns
          const int kind = __shfl_sync(0xffffffffu, t_kind, u - ub);
          const int len = __shfl_sync(0xffffffffu, t_len, u - ub);
          if (kind) {
            if (j >= e) return -1;
            int sn, f2;
            stream_geom(len, &sn, &f2);
            return j < sn ? j : f2 + (j - sn);
          }
        }
        if (j >= e) return -1;
        return a.idx[static_cast<size_t>(row) * istride + j];
      };
      // raw page-table entry of a position inside the request, -1 outside
      // whether position pos lies inside unit u's request (its page-table entry is then read and
      // must name a physical page: a bad entry, negative or too large, raises the status)
      auto pos_in = [&](int u, int pos) -> bool {
        if (u >= ue) return false;
        const int len = __shfl_sync(0xffffffffu, t_len, u - ub);
        return pos >= 0 && pos < (len + page - 1) / page;
      };
      auto load_phys = [&](int u, int pos) -> int {
        if (u >= ue) return -1;
        const int row = __shfl_sync(0xffffffffu, t_row, u - ub);
        const int len = __shfl_sync(0xffffffffu, t_len, u - ub);
        const int b = row / kv.Hkv;
        const int npos = (len + page - 1) / page;
        return pos >= 0 && pos < npos ? kv.page_table[static_cast<size_t>(b) * kv.max_pages + pos]
                                      : -1;
      };
      int ua, ba, ubb, bb, uc, bc;
      seek(ub, ub == 0 && f_beg >= 0 ? f_beg : __shfl_sync(0xffffffffu, t_beg, 0), &ua, &ba);
      seek(ua, ba + 32, &ubb, &bb);
      int pos_a = load_sel(ua, ba), pos_b = load_sel(ubb, bb);
      for (; uq <= ua && uq < ue && !stopped; ++uq) stopped = !publish(uq);
      DSA_STAMP_DIRECT(g_trace_stream, 11, kSW * 32 + (pos_a == -12345));
      int raw_a = load_phys(ua, pos_a);
      bool in_a = pos_in(ua, pos_a);
      while (ua < ue && !stopped) {
        seek(ubb, bb + 32, &uc, &bc);
        const int pos_c = load_sel(uc, bc);
        const int raw_b = load_phys(ubb, pos_b);
        const bool in_b = pos_in(ubb, pos_b);
        for (; uq <= ua && uq < ue && !stopped; ++uq) stopped = !publish(uq);
        if (stopped) break;
        // issue chunk A
        const int row = __shfl_sync(0xffffffffu, t_row, ua - ub);
        const int e = __shfl_sync(0xffffffffu, t_end, ua - ub);
        const int h = row % kv.Hkv;
        const int nb = min(32, e - ba);
        const bool in_range = in_a;  // position inside the request
        const bool ok = in_range && raw_a >= 0 && raw_a < kv.num_phys;
        if (in_range && !ok) raise_status(kv.status, DSA_STATUS_BAD_PAGE);
        for (int q0 = 0; q0 < nb; q0 += NL) {
          const int src = min(31, q0 + (lane < NL ? lane : 0));
          const int pk = __shfl_sync(0xffffffffu, pos_a, src);
          const int phk = __shfl_sync(0xffffffffu, raw_a, src);
          const int okk = __shfl_sync(0xffffffffu, ok ? 1 : 0, src);
          const bool active = lane < NL && q0 + lane < nb;
          const int ii = i + q0 + lane;
          const int s = ii % S, uu = ii / S;
          int stop = 0;
          if (active && uu > 0 &&
              !mbar_wait(smem_u32(&bars[S + s]), (uu - 1) & 1, abort_flag, kv.status))
            stop = 1;
          if (__any_sync(0xffffffffu, stop)) {  // the whole warp leaves together
            stopped = true;
            break;
          }
          if (active) {
            const uint32_t full = smem_u32(&bars[s]);
            stage_pos[s] = pk;
            stage_ok[s] = okk;  // both published by the arrive below
            if (!okk) {
              mbar_arrive(full);  // nothing to load: complete the phase with a plain arrival
            } else {
              const uint32_t dst = smem_base + s * stage_bytes;
              const int row0 = (phk * kv.Hkv + h) * page;
              mbar_arrive_expect_tx(full, stage_tx);
              if (QNT) {  // the page's block (K and V codes, their scales): one bulk copy
                bulk_load(dst, a.qkv + static_cast<size_t>(row0) * kBpt, kBpt * page, full);
              } else {
                tma_load_page(dst, &tmK, row0, full);
                tma_load_page(dst + 2 * page * 128, &tmV, row0, full);
              }
            }
          }
          if (lane == 0) *issued = i + min(nb, q0 + NL);
          DSA_STAMP_DIRECT(g_trace_stream, 18, kSW * 32);  // the loop's first loads issued
        }
        i += nb;
        ua = ubb;
        ba = bb;
        pos_a = pos_b;
        raw_a = raw_b;
        in_a = in_b;
        ubb = uc;
        bb = bc;
        pos_b = pos_c;
      }
      for (; uq < ue && !stopped; ++uq) stopped = !publish(uq);  // units without pages
    }
    __syncwarp();
    if (lane == 0) *producer_done = 1;
    DSA_STAMP_DIRECT(g_trace_stream, 9, kSW * 32);  // producer: every load issued
    return;  // the producer takes no part in the epilogues (they use named barrier 1)
  }

  // ---- consumers: warp `warp` owns tile t of stage s when (s * tiles + t) % kSW == warp
  uint64_t own_stages = 0;
  for (int s = 0; s < S; ++s)
    if (((warp - s * tiles) % kSW + kSW) % kSW < tiles) own_stages |= 1ull << s;
  int i = 0;  // ring position, in lock-step with the producer
  bool any_cut = false;
  // Unit u = n_units is a rehearsal: it runs the unit epilogue and the cut-row merge (the same
  // instructions) with every global write suppressed, so that the merge code is in L2 when the
  // CTAs that take the rows' last tickets reach it (after an L2 flush it would otherwise come from
  // HBM there, on the launch's critical path).  Only CTAs holding a single unit and merging nothing
  // rehearse: they finish well before the CTAs holding two units, which run one more epilogue and
  // take the last tickets, so the rehearsal's own cold fetches cost the launch nothing.
  bool merged = false;  // this CTA merged a cut row (uniform across the consumer warps)
#ifdef DSA_TIMELINE
  int n_owned = 0;  // pages this warp has taken (for the per-page stamps)
#endif
  const int n_iter = n_units + (n_units == 1 ? 1 : 0);
  // The geometry of the rows this CTA may share with others (its first and its last unit), worked
  // out now, while the first pages are on their way: at the end only the tickets remain.
  int* cut_info = misc + 20;  // [2][first CTA, CTA count, row, record slot of the first CTA]
  if (warp == 0 && lane < 2) {
    const int di = d_first + (lane == 0 ? 0 : n_units - 1);
    const long long rs = unit_start(di);
    const int c_first = slot_owner(rs, T, n_act);
    const int c_last = slot_owner(rs + unit_stride(di) - 1, T, n_act);
    cut_info[lane * 4 + 0] = c_first;
    cut_info[lane * 4 + 1] = c_last - c_first + 1;
    cut_info[lane * 4 + 2] = unit_row(di);
    // the row is the first CTA's last unit: slot 1 unless it is also that CTA's first
    cut_info[lane * 4 + 3] = slot_start(c_first, T, n_act) < rs ? 1 : 0;
  }
  for (int u = 0; u < n_iter; ++u) {
    const bool dry = u == n_units;
    if (dry && merged) break;
    const int slot = u & 1;
    const bool got =
        !dry && mbar_wait(smem_u32(&qbars[slot]), (u >> 1) & 1, abort_flag, kv.status);
    const int row = dry ? 0 : desc[slot * 4 + 0];
    const int beg = dry ? 0 : desc[slot * 4 + 1];
    const int end = got ? desc[slot * 4 + 2] : beg;
    const int L = dry ? 0 : desc[slot * 4 + 3];
    const bool strm = STREAMING && !dry && desc_kind[slot] != 0;
    // a streaming unit attends only tokens [0, sink) and [L - local, L) of its pages
    const int lo_end = strm ? min(a.sink, L) : L, hi_beg = strm ? max(0, L - a.local) : 0;
    const int b = row / kv.Hkv, h = row % kv.Hkv;
    const int di = d_first + u;
    uint32_t qa[8][4] = {};
    if (!dry) {
      if (TR && KV4)
        load_qT_frags_kv4(sQ + slot * 16 * kHeadDim, qa);
      else if (TR && KV8)
        load_qT_frags(sQ + slot * 16 * kHeadDim, qa);
      else if (TR)
        load_qT_frags_bf16(sQ + slot * 16 * kHeadDim, qa);
      else if (QNT)
        load_q_frags_kv8(sQ + slot * 16 * kHeadDim, qa);
      else
        load_q_frags(sQ + slot * 16 * kHeadDim, qa, kHeadDim);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&qbars[2 + slot]));
    }
    DSA_STAMP_DIRECT(g_trace_stream, 2, 0);  // first unit's descriptor and query on chip
    std::conditional_t<TR, WarpStateT, WarpSoftmaxState> st;
    state_init(st);
    const int npg = end - beg;
    // stage and phase parity of ring position i + k, stepped along without divisions (a warp
    // passes over the positions of stages it does not own many times per page)
    int s_next = i % S, ph_next = (i / S) & 1;
    for (int k = 0; k < npg; ++k) {
      const int s = s_next, ph = ph_next;
      if (++s_next == S) {
        s_next = 0;
        ph_next ^= 1;
      }
      if (!((own_stages >> s) & 1ull)) continue;
#ifdef DSA_TIMELINE
      const int owned_k = n_owned++;  // warp 0's fourth page of its first unit, timed alone
      DSA_STAMP_DIRECT(g_trace_stream, 24, owned_k == 3 ? 0 : 1 << 20);
#endif
      if (!mbar_wait(smem_u32(&bars[s]), ph, abort_flag, kv.status)) break;
      DSA_STAMP_DIRECT(g_trace_stream, 3, 0);  // warp 0's first page landed
      DSA_STAMP_DIRECT(g_trace_stream, 22, owned_k == 3 ? 0 : 1 << 20);
      const int pos = stage_pos[s];
      const bool loaded = stage_ok[s] != 0;
      const uint32_t kb = smem_base + s * stage_bytes;
      const uint32_t vb = kb + 2 * page * 128;
      bool wrote = false;
      int arrivals = 0;
      for (int t = ((warp - s * tiles) % kSW + kSW) % kSW; t < tiles; t += kSW) {
        ++arrivals;
        if (!loaded) continue;
        const int tok = pos * page + t * 16 + (lane & 15);
        const bool in = tok < L && (tok < lo_end || tok >= hi_beg);
        const uint32_t vm = __ballot_sync(0xffffffffu, in) & 0xffffu;
        if (vm == 0u) continue;
        if constexpr (TR && !QNT) {
          if (vm != 0xffffu)
            wrote |=
                zero_invalid_v_rows(vm, smem + s * stage_bytes + 2 * page * 128, page, t * 16);
          float sc4[4];
          tileT_scores_bf16(qa, kb, page, t * 16, sc4);
          tileT_softmax_pv_bf16(st, sc4, a.scale_log2, vm, vb, page, t * 16);
          continue;
        } else if constexpr (TR) {
          const uint8_t* blk = smem + s * stage_bytes;  // the page's quantised block
          const int rowb = KV8 ? 128 : 64;  // bytes per code row
          const float* ksc = reinterpret_cast<const float*>(blk + 2 * rowb * page) + t * 16;
          float sc4[4];
          tileT_scores<FMT>(qa, blk + t * 16 * rowb, sc4);
          tileT_softmax_pv<FMT>(st, sc4, a.scale_log2, vm, blk + (page + t * 16) * rowb, ksc,
                                ksc + page);
          continue;
        } else {
        float sc[2][4];
        if (KV8) {
          const uint8_t* blk = smem + s * stage_bytes;  // the page's KV8 block
          const float* ksc = reinterpret_cast<const float*>(blk + 256 * page) + t * 16;
          tile_scores_kv8(qa, blk + t * 16 * 128, sc);
          tile_softmax_pv_q<kFmtKv8>(st, sc, a.scale_log2, vm, blk + (page + t * 16) * 128, ksc,
                                     ksc + page);
        } else if (KV4) {
          const uint8_t* blk = smem + s * stage_bytes;  // the page's KV4 block
          const float* ksc = reinterpret_cast<const float*>(blk + 128 * page) + t * 16;
          tile_scores_kv4(qa, blk + t * 16 * 64, sc);
          tile_softmax_pv_q<kFmtKv4>(st, sc, a.scale_log2, vm, blk + (page + t * 16) * 64, ksc,
                                     ksc + page);
        } else {
          if (vm != 0xffffu)
            wrote |=
                zero_invalid_v_rows(vm, smem + s * stage_bytes + 2 * page * 128, page, t * 16);
          tile_scores(qa, kb, page, t * 16, sc);
          tile_softmax_pv(st, sc, a.scale_log2, vm, vb, page, t * 16);
        }
        }
      }
      if (wrote) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        for (int r = 0; r < arrivals; ++r) mbar_arrive(smem_u32(&bars[S + s]));
      DSA_STAMP_DIRECT(g_trace_stream, 23, owned_k == 3 ? 0 : 1 << 20);
    }
    i += npg;
    DSA_STAMP_DIRECT(g_trace_stream, 4, 0);  // warp 0 through the first unit's pages
    state_finish(st);

    // ---- unit epilogue: merge the warps' states of the G query heads
    if constexpr (TR) {
      const int g8 = lane >> 2, q0 = (lane & 3) * 2;
      float* wO = sO + warp * G * kHeadDim;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        if constexpr (QNT) {  // lane (g, tig): dims 16 g + 2 mt, + 1 of heads 2 tig, 2 tig + 1
          const int d = 16 * g8 + 2 * mt;
          if (q0 < G)
            *reinterpret_cast<float2*>(wO + q0 * kHeadDim + d) =
                make_float2(st.o[mt][0], st.o[mt][2]);
          if (q0 + 1 < G)
            *reinterpret_cast<float2*>(wO + (q0 + 1) * kHeadDim + d) =
                make_float2(st.o[mt][1], st.o[mt][3]);
        } else {  // lane (g, tig): dims 16 mt + g, + 8 of heads 2 tig, 2 tig + 1
          const int d = 16 * mt + g8;
          if (q0 < G) {
            wO[q0 * kHeadDim + d] = st.o[mt][0];
            wO[q0 * kHeadDim + d + 8] = st.o[mt][2];
          }
          if (q0 + 1 < G) {
            wO[(q0 + 1) * kHeadDim + d] = st.o[mt][1];
            wO[(q0 + 1) * kHeadDim + d + 8] = st.o[mt][3];
          }
        }
      }
      if (g8 == 0) {
        if (q0 < G) {
          sM[warp * G + q0] = st.m[0];
          sL[warp * G + q0] = st.l[0];
        }
        if (q0 + 1 < G) {
          sM[warp * G + q0 + 1] = st.m[1];
          sL[warp * G + q0 + 1] = st.l[1];
        }
      }
    } else {
      const int r0 = lane >> 2, c0 = (lane & 3) * 2;
      float* wO = sO + warp * G * kHeadDim;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (QNT) {  // column c of n-tile j is dim 16 c + j
          if (r0 < G) {
            wO[r0 * kHeadDim + kv8_o_pos(r0, 16 * c0 + j)] = st.o[j][0];
            wO[r0 * kHeadDim + kv8_o_pos(r0, 16 * c0 + 16 + j)] = st.o[j][1];
          }
          if (r0 + 8 < G) {
            wO[(r0 + 8) * kHeadDim + kv8_o_pos(r0 + 8, 16 * c0 + j)] = st.o[j][2];
            wO[(r0 + 8) * kHeadDim + kv8_o_pos(r0 + 8, 16 * c0 + 16 + j)] = st.o[j][3];
          }
          continue;
        }
        if (r0 < G)
          *reinterpret_cast<float2*>(wO + r0 * kHeadDim + j * 8 + c0) =
              make_float2(st.o[j][0], st.o[j][1]);
        if (r0 + 8 < G)
          *reinterpret_cast<float2*>(wO + (r0 + 8) * kHeadDim + j * 8 + c0) =
              make_float2(st.o[j][2], st.o[j][3]);
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
    named_barrier(1, kSConsumers);
    DSA_STAMP_DIRECT(g_trace_stream, 14, u == n_units - 1 ? 0 : 1 << 20);  // last unit's pages
    // cut: the unit reaches outside this CTA's slot range (other CTAs hold part of the row)
    const long long rs = dry ? my_beg : unit_start(di);
    const bool cut = !dry && (rs < my_beg || rs + unit_stride(di) > my_end);
    any_cut |= cut;
    float* rec0 =
        a.part + (static_cast<size_t>(blockIdx.x) * 2 + (u == 0 ? 0 : 1)) * G * kRecordFloats;
    // Merge weights first: thread g * kSW + w takes warp w's (m, l) of head g; the kSW threads of a
    // head (consecutive lanes) reduce the maximum and the denominator with shuffles and leave
    // exp2(m_w - M) / L_total in place of m_w.  The head's own (m, l) are written here too.
    if (warp < (kSW * G + 31) / 32) {
      const int g = tid / kSW, w = tid % kSW;
      const bool mine = g < G;
      const float mw = mine ? sM[w * G + g] : -INFINITY;
      float M = mw;
#pragma unroll
      for (int o = 1; o < kSW; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
      float Lsum = mine ? sL[w * G + g] * f : 0.f;
#pragma unroll
      for (int o = 1; o < kSW; o <<= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
      if (mine) sM[w * G + g] = Lsum > 0.f ? __fdividef(f, Lsum) : 0.f;
      const float mn = Lsum > 0.f ? M * kLn2 : -INFINITY;
      if (mine && w == 0 && !dry) {
        if (!cut) {
          const size_t qh = static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G + g;
          a.m[qh] = mn;
          a.l[qh] = Lsum;
        } else {
          rec0[g * kRecordFloats + 128] = mn;
          rec0[g * kRecordFloats + 129] = Lsum;
        }
      }
    }
    named_barrier(1, kSConsumers);
    for (int e = tid; e < G * kHeadDim; e += kSConsumers) {
      const int g = e >> 7, d = e & 127;
      const int pos = QNT && !TR ? kv8_o_pos(g, d) : d;
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kSW; ++w) o += sO[(w * G + g) * kHeadDim + pos] * sM[w * G + g];
      if (!dry && !cut)  // the rehearsal writes nothing
        a.out[(static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G + g) * kHeadDim + d] = o;
      else if (!dry)
        rec0[g * kRecordFloats + d] = o;
    }
    DSA_STAMP_DIRECT(g_trace_stream, 20, u == n_units - 1 ? 0 : 1 << 20);  // thread 0's part
    named_barrier(1, kSConsumers);  // the merge area is rewritten by the next unit
    DSA_STAMP_DIRECT(g_trace_stream, 5, 0);  // the first unit's epilogue done
    DSA_STAMP_DIRECT(g_trace_stream, 15, u == n_units - 1 ? 0 : 1 << 20);  // the last one's

    // ---- rows cut across CTAs (only this CTA's first and last units can be).  Both tickets are
    // taken at once when all of this CTA's records are written; the CTA that takes a row's last
    // ticket merges the row's records in CTA order, eight records per round trip, one query head
    // per warp.  The row's record geometry (first CTA, CTA count, the first CTA's record slot) is
    // worked out once per cut row, beside its ticket: the merge itself divides nothing.
    // (In the rehearsal both "cut rows" are this CTA's own record slot 0, marked last, and nothing
    // is written to global memory or counted; its unit epilogue writes nothing either.)
    if (dry || (u == n_units - 1 && any_cut)) {
      const int n_cut = dry || n_units > 1 ? 2 : 1;
      if (dry && warp == 0 && lane < 2) {
        cut_info[lane * 4 + 0] = blockIdx.x;
        cut_info[lane * 4 + 1] = 1;
        cut_info[lane * 4 + 2] = 0;
        cut_info[lane * 4 + 3] = 0;
        last_flag[lane] = 1;
      } else if (!dry && warp == 0 && lane < n_cut) {
        const int C = cut_info[lane * 4 + 1];
        const int last = C > 1 && ticket_add(a.counters + cut_info[lane * 4 + 2]) == C - 1;
        last_flag[lane] = last;
        DSA_STAMP_DIRECT(g_trace_stream, 21, last == -12345 ? 1 << 20 : 0);  // ticket returned
      }
      named_barrier(1, kSConsumers);
      if (!dry) merged = last_flag[0] != 0 || (n_cut > 1 && last_flag[1] != 0);
      DSA_STAMP_DIRECT(g_trace_stream, 16, dry ? 1 << 20 : 0);  // tickets taken
      const int n_jobs = n_cut * G;  // (cut row, head) pairs
      for (int job = warp; job < n_jobs; job += kSW) {
        const int k = job / G, g = job - k * G;
        if (!last_flag[k]) continue;
        const int c_first = cut_info[k * 4 + 0];
        const int C = cut_info[k * 4 + 1];
        const int row = cut_info[k * 4 + 2];
        const int slot_first = cut_info[k * 4 + 3];
        float M = -INFINITY, Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < C; c0 += 8) {
          float4 v[8];
          float mv[8], lv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            mv[j] = -INFINITY;
            lv[j] = 0.f;
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int c = c_first + c0 + j;
            if (c0 + j < C) {
              const int slot = c0 + j == 0 ? slot_first : 0;  // later CTAs start inside the row
              const float* r =
                  a.part + ((static_cast<size_t>(c) * 2 + slot) * G + g) * kRecordFloats;
              v[j] = __ldcg(reinterpret_cast<const float4*>(r) + lane);
              mv[j] = __ldcg(r + 128);
              lv[j] = __ldcg(r + 129);
            }
          }
          float Mn = M;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (lv[j] > 0.f) Mn = fmaxf(Mn, mv[j]);
          if (Mn == -INFINITY) continue;
          const float f = M == -INFINITY ? 0.f : fast_exp2((M - Mn) * kLog2e);
          Ls *= f;
          acc.x *= f;
          acc.y *= f;
          acc.z *= f;
          acc.w *= f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float wgt = lv[j] > 0.f ? lv[j] * fast_exp2((mv[j] - Mn) * kLog2e) : 0.f;
            Ls += wgt;
            acc.x += wgt * v[j].x;
            acc.y += wgt * v[j].y;
            acc.z += wgt * v[j].z;
            acc.w += wgt * v[j].w;
          }
          M = Mn;
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const int b = row / kv.Hkv, h = row % kv.Hkv;
        const size_t qh = static_cast<size_t>(b) * kv.Hq + static_cast<size_t>(h) * G + g;
        if (dry) continue;
        *reinterpret_cast<float4*>(a.out + qh * kHeadDim + lane * 4) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (lane == 0) {
          a.m[qh] = Ls > 0.f ? M : -INFINITY;
          a.l[qh] = Ls;
          if (g == 0) a.counters[row] = 0;  // ready for the next call
        }
      }
      DSA_STAMP_DIRECT(g_trace_stream, 17, !dry && merged ? 0 : 1 << 20);  // merge done
    }
  }

  DSA_STAMP_DIRECT(g_trace_stream, 6, 0);  // the consumers' work done (end)
  // after a timeout, wait (bounded) for the page loads still in flight before the CTA exits
  if (tid == 0 && *abort_flag) {
    const unsigned long long t0 = global_timer_ns();
    while (!*producer_done && global_timer_ns() - t0 < 50000000ull) {
    }
    const int n = *issued;
    for (int k = max(0, n - S); k < n; ++k)
      if (!mbar_wait_drain(smem_u32(&bars[k % S]), (k / S) & 1)) break;
  }
}

}  // namespace

size_t stream_attn_smem_bytes(int page, int stages, int G, int qbits) {
  return slayout(page, stages, G, qbits).total;
}

int stream_attn_grid() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return kStreamMaxGrid;
  return sms < kStreamMaxGrid ? sms : kStreamMaxGrid;
}

cudaError_t launch_stream_attn(const CUtensorMap& tmK, const CUtensorMap& tmV,
                               const StreamAttnArgs& a, int grid, cudaStream_t s) {
  const int fmt = a.qkv != nullptr ? a.qbits : kFmtBf16;
  const size_t bytes = slayout(a.kv.p, a.stages, a.kv.G, fmt).total;
  auto go = [&](auto kernel) -> cudaError_t {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, grid, kSThreads, bytes, s, tmK, tmV, a);
  };
  // the transposed tiles when the query group fits their n8 columns
  const bool tr = a.kv.G <= 8;
  if (fmt == kFmtKv8)
    return tr ? go(stream_attn_kernel<false, kFmtKv8, true>) : go(stream_attn_kernel<false, kFmtKv8>);
  if (fmt == kFmtKv4)
    return tr ? go(stream_attn_kernel<false, kFmtKv4, true>) : go(stream_attn_kernel<false, kFmtKv4>);
  if (a.stream_stride > 0)
    return tr ? go(stream_attn_kernel<true, kFmtBf16, true>) : go(stream_attn_kernel<true, kFmtBf16>);
  return tr ? go(stream_attn_kernel<false, kFmtBf16, true>) : go(stream_attn_kernel<false, kFmtBf16>);
}

}  // namespace dsa

#ifdef DSA_TIMELINE
// Phase-trace accessors of the traced library (see DSA_TRACE_BEGIN).
extern "C" int dsa_trace_read_stream(void* host, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(
      host, dsa::g_trace_stream,
      bytes < sizeof(dsa::g_trace_stream) ? bytes : sizeof(dsa::g_trace_stream)));
}
extern "C" int dsa_trace_clear_stream() {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, dsa::g_trace_stream);
  return static_cast<int>(e == cudaSuccess ? cudaMemset(p, 0, sizeof(dsa::g_trace_stream)) : e);
}
#endif
