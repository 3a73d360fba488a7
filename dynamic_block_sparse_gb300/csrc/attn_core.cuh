// Per-warp attention over one 16-token tile of a KV page staged in shared memory.
//
// A page of p tokens is staged as four TMA boxes (SWIZZLE_128B): K dims 0..63, K dims 64..127,
// V dims 0..63, V dims 64..127, each p rows of 128 bytes.  A warp owns the whole query group of a
// KV head as the M = 16 rows of mma.m16n8k16 (rows >= G are zero), so each K/V byte is read from
// HBM once per KV head:
//   S[16 x 16 tokens]  = Q[16 x 128] . K_tile^T      (8 k-steps x 2 n-tiles)
//   online softmax over the tile (log2 domain), P rounded to bf16 in registers
//   O[16 x 128]       += P[16 x 16] . V_tile[16 x 128] (16 n-tiles)
// Logits are s = scale * q.k; the running max is kept as scale*log2(e)*q.k.
#pragma once

#include "common.cuh"

namespace dsa {

constexpr int kQStride = 136;  // bf16 elements per staged query row (272 B: conflict-free reads)

struct WarpSoftmaxState {
  float o[16][4];  // O accumulator fragments: n-tile j covers dims 8j..8j+7
  float m[2];      // running max (log2 units) of rows lane/4 and lane/4 + 8
  float l[2];      // thread-partial denominators of the same rows
};

DSA_DEV void state_init(WarpSoftmaxState& st) {
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[j][e] = 0.f;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.f;
}

// A-operand fragments of the staged query tile (sQ: 16 rows of `stride` bf16).
DSA_DEV void load_q_frags(const __nv_bfloat16* sQ, uint32_t (&qa)[8][4], int stride = kQStride) {
  const int lane = threadIdx.x & 31;
  const int r0 = lane >> 2, c0 = (lane & 3) * 2;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c = ks * 16 + c0;
    qa[ks][0] = *reinterpret_cast<const uint32_t*>(sQ + r0 * stride + c);
    qa[ks][1] = *reinterpret_cast<const uint32_t*>(sQ + (r0 + 8) * stride + c);
    qa[ks][2] = *reinterpret_cast<const uint32_t*>(sQ + r0 * stride + c + 8);
    qa[ks][3] = *reinterpret_cast<const uint32_t*>(sQ + (r0 + 8) * stride + c + 8);
  }
}

// S = Q . K_tile^T for tokens [row0, row0 + 16) of a staged page.
// kbase: shared address of the K box for dims 0..63; the dims 64..127 box follows at +page*128.
DSA_DEV void tile_scores(const uint32_t (&qa)[8][4], uint32_t kbase, int page, int row0,
                         float (&sc)[2][4]) {
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3;
  const uint32_t tok = static_cast<uint32_t>(row0 + (mi >> 1) * 8 + (lane & 7));
  // two independent accumulation chains per n-tile (even / odd k-steps) halve the mma latency
  float acc[2][2][4];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[c][nt][e] = 0.f;
  const uint32_t half_stride = static_cast<uint32_t>(page * 128);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t chunk = static_cast<uint32_t>(ks * 2 + (mi & 1));
    const uint32_t addr = kbase + (chunk >> 3) * half_stride + sw128(tok, chunk & 7u);
    uint32_t b0, b1, b2, b3;
    ldsm_x4(addr, b0, b1, b2, b3);
    mma_bf16(acc[ks & 1][0], qa[ks], b0, b1);
    mma_bf16(acc[ks & 1][1], qa[ks], b2, b3);
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[nt][e] = acc[0][nt][e] + acc[1][nt][e];
}

// Online-softmax update with the tile's logits (raw q.k in sc), then O += P . V_tile.
// `valid` has bit t set when token row0 + t takes part.
DSA_DEV void tile_softmax_pv(WarpSoftmaxState& st, float (&sc)[2][4], float scale_log2,
                             uint32_t valid, uint32_t vbase, int page, int row0) {
  const int lane = threadIdx.x & 31;
  const int tig = lane & 3;
  float x[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = nt * 8 + tig * 2 + (e & 1);
      x[nt][e] = ((valid >> col) & 1u) ? sc[nt][e] * scale_log2 : -INFINITY;
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
  // once the running maxima settle the rescale is a no-op for the whole warp: skip it
  if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      st.o[j][0] *= alpha[0];
      st.o[j][1] *= alpha[0];
      st.o[j][2] *= alpha[1];
      st.o[j][3] *= alpha[1];
    }
  }
  uint32_t pa[4];
  pa[0] = pack_bf16(p[0][0], p[0][1]);
  pa[1] = pack_bf16(p[0][2], p[0][3]);
  pa[2] = pack_bf16(p[1][0], p[1][1]);
  pa[3] = pack_bf16(p[1][2], p[1][3]);
  const int mi = lane >> 3;
  const uint32_t tok = static_cast<uint32_t>(row0 + (mi & 1) * 8 + (lane & 7));
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) {
    const uint32_t chunk = static_cast<uint32_t>(jj * 2 + (mi >> 1));
    const uint32_t addr = vbase + (chunk >> 3) * static_cast<uint32_t>(page * 128) +
                          sw128(tok, chunk & 7u);
    uint32_t v0, v1, v2, v3;
    ldsm_x4_t(addr, v0, v1, v2, v3);
    mma_bf16(st.o[2 * jj], pa, v0, v1);
    mma_bf16(st.o[2 * jj + 1], pa, v2, v3);
  }
}

// Zeroes the V rows of tokens that do not take part, so that stale pool contents (possibly
// NaN/Inf) never reach the P.V product.  Returns true if anything was written.
DSA_DEV bool zero_invalid_v_rows(uint32_t valid, uint8_t* vtile, int page, int row0) {
  const int lane = threadIdx.x & 31;
  bool wrote = false;
  if (lane < 16 && !((valid >> lane) & 1u)) {
    uint4 z = make_uint4(0, 0, 0, 0);
    uint4* a = reinterpret_cast<uint4*>(vtile + (row0 + lane) * 128);
    uint4* b = reinterpret_cast<uint4*>(vtile + page * 128 + (row0 + lane) * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      a[c] = z;
      b[c] = z;
    }
    wrote = true;
  }
  __syncwarp();
  return wrote;
}

// Finishes the thread-partial denominators (sum over the 4 lanes holding a row).
DSA_DEV void state_finish(WarpSoftmaxState& st) {
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 1);
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 2);
  }
}

// Writes a warp's (unnormalised O, m, l) to shared scratch: sO [16][128] fp32, sM/sL [16].  Only
// the first `rows` query rows of O are written (the rest are padding).
DSA_DEV void state_store(const WarpSoftmaxState& st, float* sO, float* sM, float* sL,
                         int rows = 16) {
  const int lane = threadIdx.x & 31;
  const int r0 = lane >> 2, c0 = (lane & 3) * 2;
  if (r0 < rows) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *reinterpret_cast<float2*>(sO + r0 * 128 + j * 8 + c0) = make_float2(st.o[j][0], st.o[j][1]);
  }
  if (r0 + 8 < rows) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *reinterpret_cast<float2*>(sO + (r0 + 8) * 128 + j * 8 + c0) =
          make_float2(st.o[j][2], st.o[j][3]);
  }
  if ((lane & 3) == 0) {
    sM[r0] = st.m[0];
    sM[r0 + 8] = st.m[1];
    sL[r0] = st.l[0];
    sL[r0 + 8] = st.l[1];
  }
}

// ------------------------------------------------------------------------------- page lists

DSA_DEV bool contains_sorted(const int32_t* a, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int v = a[mid];
    if (v == x) return true;
    if (v < x) lo = mid + 1;
    else hi = mid;
  }
  return false;
}

// Appends the valid candidates of one warp-wide round to the list, preserving order.
DSA_DEV int append_round(bool ok, int phys, int pos, int2* list, int n) {
  const int lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xffffffffu, ok);
  if (ok) {
    const int at = n + __popc(bal & ((1u << lane) - 1u));
    if (at < kMaxListPages) list[at] = make_int2(phys, pos);
  }
  return n + __popc(bal);
}

// Page table lookup of position `pos` of request b, with range checks.
DSA_DEV bool lookup_page(const KvView& kv, int b, int pos, int npos, int* phys) {
  if (pos < 0 || pos >= npos) return false;
  const int ph = kv.page_table[static_cast<size_t>(b) * kv.max_pages + pos];
  if (ph < 0 || ph >= kv.num_phys) {
    raise_status(kv.status, DSA_STATUS_BAD_PAGE);
    return false;
  }
  *phys = ph;
  return true;
}

}  // namespace dsa
