// swiglu.cu -- the gate between the stacked gate/up projection and the down
// projection of a SwiGLU MLP block, and its backward:
//
//     h  = silu(g) * u,               silu(x) = x * sigma(x) = x / (1 + e^-x)
//     dg = dh * u * sigma(g) * (1 + g * (1 - sigma(g)))
//     du = dh * silu(g)
//
// The pages fuse the MLP of the transformer block into their forward
// ("Unsloth性能实测：比传统方法快2倍真的吗？", section 2.2) and name SwiGLU among the
// fused transformer operators ("UnSloth加速原理：CUDA内核融合与内存优化", section
// "在ms-swift中的角色").
//
// Layout: gu [M, 2*d_ff] is the stacked projection's output, gate columns
// [0, d_ff) then up columns [d_ff, 2*d_ff) -- or, interleaved, 64-column
// chunks [gate 0..63 | up 0..63 | gate 64..127 | ...], the layout whose gate
// the main kernel's epilogue computes; h and dh are [M, d_ff]; the
// backward writes dgu in the layout of gu, which is the dY of the stacked
// projection's backward.  All bf16; the arithmetic is fp32 with one rounding
// of each output.  HBM-bound: 6 B per h element forward, 10 B backward.

#include <cuda_bf16.h>
#include <cstdint>

#include "kernels.h"

namespace qlora {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float sigmoid(float x) { return 1.f / (1.f + expf(-x)); }

// Column of gate feature f in a row of gu; the up feature is d_ff (or, interleaved, 64) further.
__device__ __forceinline__ int64_t gate_col(int64_t f, bool interleaved) {
  return interleaved ? (f >> 6) * 128 + (f & 63) : f;
}

// One thread: 8 consecutive features of one row (16-byte loads and stores).
__global__ void __launch_bounds__(256) swiglu_fwd_kernel(const uint16_t* __restrict__ gu, int64_t rows,
                                                         int64_t d_ff, uint16_t* __restrict__ h, bool interleaved) {
  const int64_t per_row = d_ff / 8, total = rows * per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / per_row, f = (i % per_row) * 8;
    const uint16_t* row = gu + m * 2 * d_ff;
    const int64_t gc = gate_col(f, interleaved), uc = gc + (interleaved ? 64 : d_ff);
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(row + gc));
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + uc));
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float g0 = bf16_lo(gw[k]), g1 = bf16_hi(gw[k]);
      o[k] = pack2(g0 * sigmoid(g0) * bf16_lo(uw[k]), g1 * sigmoid(g1) * bf16_hi(uw[k]));
    }
    *reinterpret_cast<uint4*>(h + m * d_ff + f) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const uint16_t* __restrict__ gu,
                                                         const uint16_t* __restrict__ dh, int64_t rows,
                                                         int64_t d_ff, uint16_t* __restrict__ dgu, bool interleaved) {
  const int64_t per_row = d_ff / 8, total = rows * per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / per_row, f = (i % per_row) * 8;
    const uint16_t* row = gu + m * 2 * d_ff;
    const int64_t gc = gate_col(f, interleaved), uc = gc + (interleaved ? 64 : d_ff);
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(row + gc));
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + uc));
    const uint4 d = __ldg(reinterpret_cast<const uint4*>(dh + m * d_ff + f));
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w}, dw[4] = {d.x, d.y, d.z, d.w};
    uint32_t og[4], ou[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float dg[2], du[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float gv = e ? bf16_hi(gw[k]) : bf16_lo(gw[k]);
        const float uv = e ? bf16_hi(uw[k]) : bf16_lo(uw[k]);
        const float dv = e ? bf16_hi(dw[k]) : bf16_lo(dw[k]);
        const float sg = sigmoid(gv);
        du[e] = dv * gv * sg;
        dg[e] = dv * uv * sg * (1.f + gv * (1.f - sg));
      }
      og[k] = pack2(dg[0], dg[1]);
      ou[k] = pack2(du[0], du[1]);
    }
    uint16_t* out = dgu + m * 2 * d_ff;
    *reinterpret_cast<uint4*>(out + gc) = make_uint4(og[0], og[1], og[2], og[3]);
    *reinterpret_cast<uint4*>(out + uc) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
  }
}

// Grid-stride kernels: at most the CTAs of 256 threads that can be resident
// at once (a CTA that starts only after another has finished would run its
// share at the end, alone).
template <typename Kern>
int swiglu_grid(Kern kern, int64_t rows, int64_t d_ff) {
  int dev = 0, sms = 148, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  const int64_t want = (rows * (d_ff / 8) + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<int>(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_swiglu_fwd(const uint16_t* gu, int64_t rows, int64_t d_ff, uint16_t* h, bool interleaved,
                              cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  LaunchScope scope(kKindSwigluFwd, stream);
  swiglu_fwd_kernel<<<swiglu_grid(swiglu_fwd_kernel, rows, d_ff), 256, 0, stream>>>(gu, rows, d_ff, h, interleaved);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd(const uint16_t* gu, const uint16_t* dh, int64_t rows, int64_t d_ff, uint16_t* dgu,
                              bool interleaved, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  LaunchScope scope(kKindSwigluBwd, stream);
  swiglu_bwd_kernel<<<swiglu_grid(swiglu_bwd_kernel, rows, d_ff), 256, 0, stream>>>(gu, dh, rows, d_ff, dgu, interleaved);
  return cudaGetLastError();
}

}  // namespace qlora
