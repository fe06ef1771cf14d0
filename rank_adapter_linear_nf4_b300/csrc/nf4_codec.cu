// nf4_codec.cu -- NF4 quantisation and dequantisation kernels.
//
// Quantise: each 64-element block is handled by 8 threads (8 bf16 each); the
// block absmax is a max-reduction over those 8 lanes by warp shuffles.  The
// code decision is the format's: x = fl32(w / absmax) with IEEE division,
// q = number of midpoints (c[i] + c[i+1]) / 2 strictly below x.  The
// comparison is exact: it is done against the smallest float above each
// midpoint, so "x > midpoint" and "x >= threshold" agree for every float x.
//
// Dequantise: one thread per block builds the block's 16-entry bf16 table and
// expands its 32 code bytes; the results are staged in shared memory so the
// 128 output bytes per block leave the SM as coalesced stores.  The fused
// GEMM kernels use the same table routine, so their weight operand is this
// kernel's output bit for bit.
#include <cmath>
#include <cuda_runtime.h>

#include "kernels.h"
#include "nf4_lut.cuh"

namespace qlora {

namespace {

struct Thresholds {
  float t[15];
};

Thresholds make_thresholds() {
  Thresholds th;
  for (int i = 0; i < 15; ++i) {
    const double mid =
        (static_cast<double>(kNF4LevelsHost[i]) + static_cast<double>(kNF4LevelsHost[i + 1])) * 0.5;
    const float f = static_cast<float>(mid);
    th.t[i] = (static_cast<double>(f) > mid) ? f : std::nextafter(f, INFINITY);
  }
  return th;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__global__ void __launch_bounds__(256) nf4_quantize_kernel(const uint4* __restrict__ W,
                                                          int64_t n_groups,  // n_elems / 8
                                                          uint32_t* __restrict__ packed_words,
                                                          float* __restrict__ absmax,
                                                          Thresholds th) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool active = g < n_groups;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (active) v = W[g];
  float w[8];
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[2 * i] = bf16_bits_to_float(words[i] & 0xFFFFu);
    w[2 * i + 1] = bf16_bits_to_float(words[i] >> 16);
  }
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(w[i]));
  // the 8 lanes of one block are consecutive and 8-aligned inside the warp
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));

  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = 7u;
  if (m > 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = __fdiv_rn(w[i], m);
      // q = number of thresholds <= x, found by a branch-free binary search:
      // the thresholds are ascending, so each level halves the candidate range.
      const bool b3 = x >= th.t[7];
      const float t2 = b3 ? th.t[11] : th.t[3];
      const bool b2 = x >= t2;
      const float t1 = b3 ? (b2 ? th.t[13] : th.t[9]) : (b2 ? th.t[5] : th.t[1]);
      const bool b1 = x >= t1;
      const uint32_t hi3 = (b3 ? 8u : 0u) | (b2 ? 4u : 0u) | (b1 ? 2u : 0u);   // 0,2,..,14
      // last level: threshold t[hi3] (t[14] when hi3 == 14)
      float t0 = th.t[0];
#pragma unroll
      for (int k = 2; k <= 14; k += 2) t0 = (hi3 == static_cast<uint32_t>(k)) ? th.t[k] : t0;
      q[i] = hi3 + ((x >= t0) ? 1u : 0u);
    }
  }
  uint32_t word = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) word |= ((q[2 * b] << 4) | q[2 * b + 1]) << (8 * b);
  if (active) {
    packed_words[g] = word;
    if ((threadIdx.x & 7) == 0) absmax[g >> 3] = m;
  }
}

constexpr int kDeqThreads = 256;

__global__ void __launch_bounds__(kDeqThreads) nf4_dequant_kernel(const uint4* __restrict__ packed,
                                                                 const float* __restrict__ absmax,
                                                                 int64_t n_blocks,
                                                                 uint4* __restrict__ out) {
  __shared__ uint4 stage[kDeqThreads * 8];
  const int64_t b0 = static_cast<int64_t>(blockIdx.x) * kDeqThreads;
  const int64_t b = b0 + threadIdx.x;
  if (b < n_blocks) {
    const uint4 r0 = ldg_nc_v4(packed + 2 * b);
    const uint4 r1 = ldg_nc_v4(packed + 2 * b + 1);
    const Nf4BlockTable t = nf4_block_table(ldg_nc_f32(absmax + b));
    const uint32_t words[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    const int row = threadIdx.x;
#pragma unroll
    for (int c = 0; c < 8; ++c) stage[row * 8 + (c ^ (row & 7))] = nf4_expand8(words[c], t);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kDeqThreads * 8; idx += kDeqThreads) {
    const int row = idx >> 3, c = idx & 7;
    if (b0 + row < n_blocks) out[(b0 + row) * 8 + c] = stage[row * 8 + (c ^ (row & 7))];
  }
}

}  // namespace

void nf4_levels_host(float out[16]) {
  for (int i = 0; i < 16; ++i) out[i] = kNF4LevelsHost[i];
}

cudaError_t launch_quantize_nf4(const uint16_t* W, int64_t n_elems, uint8_t* packed, float* absmax,
                                cudaStream_t stream) {
  static const Thresholds th = make_thresholds();
  const int64_t n_groups = n_elems / 8;
  const int64_t grid = (n_groups + 255) / 256;
  LaunchScope scope(kKindQuantize, stream);
  nf4_quantize_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(W), n_groups, reinterpret_cast<uint32_t*>(packed), absmax, th);
  return cudaGetLastError();
}

cudaError_t launch_dequant_nf4(const uint8_t* packed, const float* absmax, int64_t n_elems,
                               uint16_t* W_out, cudaStream_t stream) {
  const int64_t n_blocks = n_elems / 64;
  const int64_t grid = (n_blocks + kDeqThreads - 1) / kDeqThreads;
  LaunchScope scope(kKindDequant, stream);
  nf4_dequant_kernel<<<static_cast<unsigned>(grid), kDeqThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(packed), absmax, n_blocks, reinterpret_cast<uint4*>(W_out));
  return cudaGetLastError();
}

}  // namespace qlora
