// nf4_codec.cu -- NF4 quantisation and dequantisation kernels.
//
// Quantise: each 64-element block is handled by 8 threads (8 bf16 each); the
// block absmax is a max-reduction over those 8 lanes by warp shuffles.  The
// code decision is the format's: x = fl32(w / absmax) with IEEE division,
// q = number of midpoints (c[i] + c[i+1]) / 2 strictly below x.  The
// comparison is exact: it is done against the smallest float above each
// midpoint, so "x > midpoint" and "x >= threshold" agree for every float x.
// The quotient is formed as w times the rounded reciprocal of absmax (the same
// code for every bf16 pair; argument at the kernel), and the search is one
// table lookup per element.
//
// Dequantise: one thread per block builds the block's 16-entry bf16 table and
// expands its 32 code bytes; the results are staged in shared memory so the
// 128 output bytes per block leave the SM as coalesced stores.  The fused
// GEMM kernels use the same table routine, so their weight operand is this
// kernel's output bit for bit.
#include <algorithm>
#include <cmath>
#include <cstring>
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

// The code decision by table.  A bin of x is k = RNE(64 x + 64), read from the
// low bits of fl(x * 64 + (1.5 * 2^23 + 64)) (one rounding of an exact
// product and sum): bins are 1/64 wide, x in [-1, 1] falls in bins 0..128, and
// k is non-decreasing in x.  The thresholds are at least 0.04 apart, so a bin
// holds at most one of them, and for x in bin k
//   q = (thresholds in bins below k) + (x >= the threshold in bin k),
// exact for every float x.  Bins 129..255 only receive NaN (all-ones low
// bits): code 0, as every comparison with NaN is false.
constexpr int kBins = 256;
constexpr float kBinMagic = 12582912.0f + 64.0f;   // 1.5 * 2^23 + 64
constexpr int kTableCopies = 16;                    // lane l reads copy l % 16: no bank conflicts

struct QuantTable {
  float t[kBins];          // the threshold inside bin k, or +inf
  uint32_t q_base[kBins];  // thresholds in bins below k
};

uint32_t bin_of_host(float x) {
  const float y = std::fma(x, 64.0f, kBinMagic);
  uint32_t u;
  std::memcpy(&u, &y, sizeof(u));
  return u & 0xFFu;
}

// Empty table (q_base 0 everywhere) if two thresholds shared a bin.
QuantTable make_quant_table(const Thresholds& th, bool* ok) {
  QuantTable tab;
  *ok = true;
  for (int k = 0; k < kBins; ++k) {
    tab.t[k] = INFINITY;
    tab.q_base[k] = 0u;
  }
  uint32_t bins[15];
  for (int i = 0; i < 15; ++i) {
    bins[i] = bin_of_host(th.t[i]);
    if (bins[i] > 128u || (i > 0 && bins[i] <= bins[i - 1])) *ok = false;
  }
  if (!*ok) return tab;
  for (int k = 0; k <= 128; ++k) {
    uint32_t below = 0;
    for (int i = 0; i < 15; ++i) {
      if (bins[i] < static_cast<uint32_t>(k)) ++below;
      if (bins[i] == static_cast<uint32_t>(k)) tab.t[k] = th.t[i];
    }
    tab.q_base[k] = below;
  }
  return tab;
}

// Quantise: a persistent grid.  A chunk is 512 groups (8 elements each);
// thread i of a CTA takes groups 256 h + i of its chunks (h = 0, 1), and the
// next chunk's loads are issued before the current chunk's arithmetic.
//
// x is formed as fl(w * fl(1/m)) instead of the format's fl32(w / m).  Scaling w
// and m by the same power of two scales both quotients exactly (while fl(1/m)
// is a normal float and the quotient is not below 2^-126, where every x gives
// code 7), so every (w, m) pair is one of a pair with m in [1, 2) -- and for all
// of those, with every bf16 |w| <= m, the two give the same code (an
// exhaustive CPU check in the tests).  A block whose fl(1/m) is not a normal
// float (absmax subnormal, above 2^126 or not finite) takes the IEEE quotient
// __fdiv_rn(w, m).
constexpr int kQuantThreads = 256;
constexpr int kQuantGroupsPerThread = 2;
constexpr int kQuantChunk = kQuantThreads * kQuantGroupsPerThread;   // groups per chunk

// The 8 codes of one group (one bf16 word quadruple), packed two per byte
// (first element in the high nibble), and the block absmax.
__device__ __forceinline__ uint32_t quantize_group(const uint4 v, uint32_t tab_lane, float& absmax_out) {
  float w[8];
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[2 * i] = bf16_bits_to_float(words[i] & 0xFFFFu);
    w[2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
  }
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(w[i]));
  // the 8 lanes of one block are consecutive and 8-aligned inside the warp
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  absmax_out = m;
  if (!(m > 0.0f)) return 0x77777777u;   // all-zero block: the zero level
  const float rm = __frcp_rn(m);
  float x[8];
  if (rm >= 1.175494351e-38f && rm <= 3.402823466e38f) {   // fl(1/m) a normal float
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(w[i], rm);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __fdiv_rn(w[i], m);
  }
  uint32_t word = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t k = __float_as_uint(__fmaf_rn(x[i], 64.0f, kBinMagic)) & 0xFFu;
    uint32_t tq0, tq1;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(tq0), "=r"(tq1) : "r"(tab_lane + k * 128u));
    // x >= t as an all-ones mask (false for NaN), so q = q_base - mask
    uint32_t ge;
    asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(ge) : "f"(x[i]), "f"(__uint_as_float(tq0)));
    const uint32_t q = tq1 - ge;
    // byte b holds code 2b in its high nibble and code 2b+1 in its low nibble
    // (the nibbles do not overlap: adding is or-ing)
    word += q << (8 * (i >> 1) + ((i & 1) ? 0 : 4));
  }
  return word;
}

__global__ void __launch_bounds__(kQuantThreads) nf4_quantize_kernel(const uint4* __restrict__ W,
                                                                    int64_t n_groups,  // n_elems / 8
                                                                    uint32_t* __restrict__ packed_words,
                                                                    float* __restrict__ absmax,
                                                                    const QuantTable table) {
  __shared__ __align__(16) uint2 s_tab[kBins * kTableCopies];
  const int64_t n_chunks = (n_groups + kQuantChunk - 1) / kQuantChunk;
  auto load_chunk = [&](int64_t c, uint4 (&v)[kQuantGroupsPerThread]) {
#pragma unroll
    for (int h = 0; h < kQuantGroupsPerThread; ++h) {
      const int64_t g = c * kQuantChunk + h * kQuantThreads + threadIdx.x;
      v[h] = (c < n_chunks && g < n_groups) ? ldg_nc_v4(W + g) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int64_t c = blockIdx.x;
  uint4 v[kQuantGroupsPerThread];
  load_chunk(c, v);
  // the table, two copies of an entry per 16-byte store
  for (int e = threadIdx.x; e < kBins * kTableCopies / 2; e += kQuantThreads) {
    const int k = e / (kTableCopies / 2);
    const uint32_t tb = __float_as_uint(table.t[k]), qb = table.q_base[k];
    reinterpret_cast<uint4*>(s_tab)[e] = make_uint4(tb, qb, tb, qb);
  }
  __syncthreads();
  const uint32_t tab_lane = smem_u32(s_tab) + static_cast<uint32_t>((threadIdx.x & (kTableCopies - 1)) * 8);
  for (; c < n_chunks; c += gridDim.x) {
    uint4 nv[kQuantGroupsPerThread];
    load_chunk(c + gridDim.x, nv);
#pragma unroll
    for (int h = 0; h < kQuantGroupsPerThread; ++h) {
      const int64_t g = c * kQuantChunk + h * kQuantThreads + threadIdx.x;
      float m;
      const uint32_t word = quantize_group(v[h], tab_lane, m);
      if (g < n_groups) {
        packed_words[g] = word;
        if ((threadIdx.x & 7) == 0) absmax[g >> 3] = m;
      }
    }
#pragma unroll
    for (int h = 0; h < kQuantGroupsPerThread; ++h) v[h] = nv[h];
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

// ---------------------------------------------------------------- the absmax in 8 bits

// One warp per group of kDqGroup block absmax values: the group's largest c
// (a shuffle max), scale2 = fl32(c / 255), and per value the nearest integer to
// fl32(a / scale2), ties to even, limited to 255 (all zero when c == 0).
__global__ void __launch_bounds__(256) absmax_dq_quantize_kernel(const float* __restrict__ absmax, int64_t n,
                                                               uint8_t* __restrict__ q8, float* __restrict__ scale2) {
  const int64_t group = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t base = group * kDqGroup;
  if (base >= n) return;   // whole warps leave together
  float v[kDqGroup / 32];
  float c = 0.0f;
#pragma unroll
  for (int j = 0; j < kDqGroup / 32; ++j) {
    const int64_t i = base + lane + 32 * j;
    v[j] = i < n ? ldg_nc_f32(absmax + i) : 0.0f;
    c = fmaxf(c, v[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, o));
  const float sc = c > 0.0f ? __fdiv_rn(c, 255.0f) : 0.0f;
#pragma unroll
  for (int j = 0; j < kDqGroup / 32; ++j) {
    const int64_t i = base + lane + 32 * j;
    if (i < n) q8[i] = sc > 0.0f ? static_cast<uint8_t>(min(255u, __float2uint_rn(__fdiv_rn(v[j], sc)))) : 0;
  }
  if (lane == 0) scale2[group] = sc;
}

// a'_i = fl32(q8_i * scale2_g).
__global__ void __launch_bounds__(256) absmax_dq_dequant_kernel(const uint8_t* __restrict__ q8,
                                                              const float* __restrict__ scale2, int64_t n,
                                                              float* __restrict__ absmax) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    absmax[i] = __fmul_rn(static_cast<float>(q8[i]), ldg_nc_f32(scale2 + i / kDqGroup));
}

}  // namespace

cudaError_t launch_quantize_absmax_dq(const float* absmax, int64_t n, uint8_t* q8, float* scale2,
                                      cudaStream_t stream) {
  const int64_t groups = (n + kDqGroup - 1) / kDqGroup;
  const int64_t grid = (groups + 7) / 8;   // 8 warps per CTA
  LaunchScope scope(kKindAbsmaxDq, stream);
  absmax_dq_quantize_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(absmax, n, q8, scale2);
  return cudaGetLastError();
}

cudaError_t launch_dequant_absmax_dq(const uint8_t* q8, const float* scale2, int64_t n, float* absmax,
                                     cudaStream_t stream) {
  // grid-stride: at most the CTAs that can be resident at once
  int dev = 0, sms = 148, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, absmax_dq_dequant_kernel, 256, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t grid = std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(sms) * per_sm);
  LaunchScope scope(kKindAbsmaxDq, stream);
  absmax_dq_dequant_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(q8, scale2, n, absmax);
  return cudaGetLastError();
}



void nf4_levels_host(float out[16]) {
  for (int i = 0; i < 16; ++i) out[i] = kNF4LevelsHost[i];
}

cudaError_t launch_quantize_nf4(const uint16_t* W, int64_t n_elems, uint8_t* packed, float* absmax,
                                cudaStream_t stream) {
  static bool table_ok = false;
  static const QuantTable table = make_quant_table(make_thresholds(), &table_ok);
  if (!table_ok) return cudaErrorInvalidValue;
  const int64_t n_groups = n_elems / 8;
  const int64_t chunks = (n_groups + kQuantChunk - 1) / kQuantChunk;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // persistent: exactly the CTAs that can be resident at once (registers, not
  // the 32 KB table, limit them), so that no CTA starts after another has finished
  static const int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nf4_quantize_kernel, kQuantThreads, 0) != cudaSuccess)
      return 1;
    return std::max(n, 1);
  }();
  const int64_t grid = std::min<int64_t>(chunks, static_cast<int64_t>(sms) * per_sm);
  LaunchScope scope(kKindQuantize, stream);
  nf4_quantize_kernel<<<static_cast<unsigned>(grid), kQuantThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(W), n_groups, reinterpret_cast<uint32_t*>(packed), absmax, table);
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
