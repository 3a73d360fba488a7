// Page scoring arithmetic shared by the scoring kernel and the fused PRR step, so that both give
// bit-identical scores (and therefore identical selections).
//
// A metadata record is 512 bytes (MINMAX: 128 x (max, min) bf16; MEAN: 128 fp32) and is read by
// a group of 8 lanes, 4 x 16 bytes each: chunk c of a record covers dims 4c..4c+3 in both
// formats, so lane (l & 7) always needs the same 16 query dims and keeps them in registers.
// The group's partial sums are combined with xor shuffles over the low three lane bits.
#pragma once

#include "common.cuh"

namespace dsa {

// Representative query of a KV head's group: the mean of its G query heads, fp32 (shared q̄[128]).
DSA_DEV void group_mean_query(const __nv_bfloat16* qg, int G, float* qbar, int tid, int nthreads) {
  for (int d = tid; d < kHeadDim; d += nthreads) {
    float s = 0.f;
    for (int r = 0; r < G; ++r) s += __bfloat162float(qg[r * kHeadDim + d]);
    qbar[d] = s / static_cast<float>(G);
  }
}

// The 16 query dims lane (l & 7) of a record group multiplies.
DSA_DEV void group_query_dims(const float* qbar, int gl, float (&qv)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) qv[i * 4 + e] = qbar[(gl + 8 * i) * 4 + e];
}

// This lane's share of one record's score (its 4 chunks).
template <int KIND>
DSA_DEV float record_partial(const uint4 (&raw)[4], const float (&qv)[16]) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (KIND == DSA_META_MINMAX) {
      const __nv_bfloat16* v = reinterpret_cast<const __nv_bfloat16*>(&raw[i]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float q = qv[i * 4 + e];
        const float hi = q * __bfloat162float(v[2 * e]);
        const float lo = q * __bfloat162float(v[2 * e + 1]);
        s += fmaxf(hi, lo);
      }
    } else {
      const float* v = reinterpret_cast<const float*>(&raw[i]);
#pragma unroll
      for (int e = 0; e < 4; ++e) s = fmaf(qv[i * 4 + e], v[e], s);
    }
  }
  return s;
}

// Loads lane gl's 4 chunks of a record.
DSA_DEV void load_record(const uint8_t* meta, size_t rec, int gl, uint4 (&raw)[4]) {
  const uint4* p = reinterpret_cast<const uint4*>(meta + rec * 512);
#pragma unroll
  for (int i = 0; i < 4; ++i) raw[i] = __ldg(p + gl + 8 * i);
}

// Sum over the 8 lanes of a record group.
DSA_DEV float group_sum(float s) {
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// ------------------------------------------------------------------------------------ EMA
// One PRR predictor update of a page's level (ell) and trend (v) from its observed score IS:
// v' = beta (IS - ell) + (1 - beta) v,  ell' = alpha IS + (1 - alpha) ell  (both from the old
// ell).  INIT, or a page with no history, starts from ell' = IS, v' = 0; a page with no score
// (past the request) gets ell' = -inf, v' = 0.
// The roundings are spelled out (one product rounded, then one fused multiply-add) so that every
// kernel computing it gives the same bits whatever the compiler would contract.
DSA_DEV void ema_step(float is, float l_old, float v_old, int mode, float alpha, float beta,
                      float& l_new, float& v_new) {
  l_new = -INFINITY;
  v_new = 0.f;
  if (is > -INFINITY) {
    if (mode == DSA_EMA_INIT || !(l_old > -INFINITY)) {
      l_new = is;
    } else {
      v_new = __fmaf_rn(beta, __fsub_rn(is, l_old), __fmul_rn(1.f - beta, v_old));
      l_new = __fmaf_rn(alpha, is, __fmul_rn(1.f - alpha, l_old));
    }
  }
}

// Predicted score ell + gamma v (-inf for pages without a score).
DSA_DEV float ema_predict(float l, float v, float gamma) {
  return l > -INFINITY ? __fmaf_rn(gamma, v, l) : -INFINITY;
}

}  // namespace dsa
