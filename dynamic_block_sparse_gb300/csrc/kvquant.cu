// Quantised KV pages: the KV pool with one fp32 scale per (page, KV head, token) row for K and one
// for V, so that every selected page the attention reads is smaller.  A (physical page, KV head)
// block is contiguous, so that one bulk copy brings a page:
//   KV8 (264 p bytes): e4m3 codes, K [p][128], V [p][128], then the K scales [p] and V scales [p].
//       Within the 128-byte code row of token slot r, the 16-byte piece of dims 16 c .. 16 c + 15
//       sits at piece c ^ (r mod 8), so that the attention's operand loads (eight rows at once)
//       hit distinct banks.
//   KV4 (136 p bytes): integer codes in [-7, 7] as offset-8 nibbles (dim 2i in the low half of
//       byte i), K [p][64], V [p][64], then the K scales [p] and V scales [p].  The 64-byte code
//       row of token r sits at row r ^ ((r >> 1) & 1) (pairs of rows swap in every other pair), so
//       that the V operand loads (rows 2i and 2i + 2 .. at once) fall in distinct bank halves.
// The quantisers; the persistent attention (stream_attn.cu) reads the codes per tile.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr float kE4m3Max = 448.f;  // largest finite e4m3 value
constexpr int kQ8Threads = 256;
constexpr int kQ8Warps = kQ8Threads / 32;

// One warp per (physical page, KV head, token) row of K (which = 0) or V (which = 1): lane l holds
// dims 4l .. 4l+3; the row's codes and scale go to their places in its block.
__global__ void __launch_bounds__(kQ8Threads)
    quantize_kv8_kernel(const __nv_bfloat16* __restrict__ src, long long n_rows, int page,
                        int which, uint8_t* __restrict__ kv8) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  const long long r = static_cast<long long>(blockIdx.x) * kQ8Warps + (threadIdx.x >> 5);
  if (r >= n_rows) return;
  const long long blk = r / page;
  const int slot = static_cast<int>(r - blk * page);
  uint8_t* base = kv8 + blk * 264 * page;
  const int lane = threadIdx.x & 31;
  const int piece = (lane >> 2) ^ (slot & 7);  // the lane's 4 dims lie in piece lane / 4
  uint8_t* dst = base + static_cast<long long>(which) * 128 * page +
                 static_cast<long long>(slot) * 128 + piece * 16 + (lane & 3) * 4;
  float* scale_out = reinterpret_cast<float*>(base + (256 + 4 * which) * page) + slot;
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(src + r * kHeadDim) + lane);
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
  float v[4];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[e] = __bfloat162float(x[e]);
    amax = fmaxf(amax, fabsf(v[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // scale: the row's largest magnitude maps to the largest e4m3 value; an all-zero row keeps 0
  const float scale = amax / kE4m3Max;
  uint32_t packed = 0u;
  if (scale > 0.f) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(v[0] / scale, v[1] / scale), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(v[2] / scale, v[3] / scale), __NV_SATFINITE, __NV_E4M3);
    packed = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  *reinterpret_cast<uint32_t*>(dst) = packed;
  if (lane == 0) *scale_out = scale;
}

constexpr int kKv4Max = 7;  // codes -7 .. 7

// One warp per (physical page, KV head, token) row of K (which = 0) or V (which = 1): lane l holds
// dims 4l .. 4l+3 and writes their two code bytes.
__global__ void __launch_bounds__(kQ8Threads)
    quantize_kv4_kernel(const __nv_bfloat16* __restrict__ src, long long n_rows, int page,
                        int which, uint8_t* __restrict__ kv4) {
  launch_dependents();  // the next kernel may be scheduled; it waits for this one
  grid_dependency_wait();  // the kernels before this one have completed
  const long long r = static_cast<long long>(blockIdx.x) * kQ8Warps + (threadIdx.x >> 5);
  if (r >= n_rows) return;
  const long long blk = r / page;
  const int slot = static_cast<int>(r - blk * page);
  const int row = slot ^ ((slot >> 1) & 1);
  uint8_t* base = kv4 + blk * 136 * page;
  const int lane = threadIdx.x & 31;
  uint8_t* dst = base + static_cast<long long>(which) * 64 * page +
                 static_cast<long long>(row) * 64 + lane * 2;
  float* scale_out = reinterpret_cast<float*>(base + (128 + 4 * which) * page) + slot;
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(src + r * kHeadDim) + lane);
  const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
  float v[4];
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    v[e] = __bfloat162float(x[e]);
    amax = fmaxf(amax, fabsf(v[e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // scale: the row's largest magnitude maps to code 7; an all-zero row keeps 0 (codes 0)
  const float scale = amax / static_cast<float>(kKv4Max);
  uint32_t nib[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    int c = 0;
    if (scale > 0.f) c = min(kKv4Max, max(-kKv4Max, __float2int_rn(v[e] / scale)));
    nib[e] = static_cast<uint32_t>(c + 8);
  }
  const uint16_t packed =
      static_cast<uint16_t>(nib[0] | (nib[1] << 4) | (nib[2] << 8) | (nib[3] << 12));
  *reinterpret_cast<uint16_t*>(dst) = packed;
  if (lane == 0) *scale_out = scale;
}

}  // namespace

cudaError_t launch_quantize_kv8(const __nv_bfloat16* src, long long n_rows, int page, int which,
                                uint8_t* kv8, cudaStream_t s) {
  const long long blocks = (n_rows + kQ8Warps - 1) / kQ8Warps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(quantize_kv8_kernel, static_cast<unsigned>(blocks), kQ8Threads, 0, s, src,
                    n_rows, page, which, kv8);
}

cudaError_t launch_quantize_kv4(const __nv_bfloat16* src, long long n_rows, int page, int which,
                                uint8_t* kv4, cudaStream_t s) {
  const long long blocks = (n_rows + kQ8Warps - 1) / kQ8Warps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(quantize_kv4_kernel, static_cast<unsigned>(blocks), kQ8Threads, 0, s, src,
                    n_rows, page, which, kv4);
}

}  // namespace dsa
