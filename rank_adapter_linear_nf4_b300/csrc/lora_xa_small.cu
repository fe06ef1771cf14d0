// lora_xa_small.cu -- T = X . A for a handful of tokens (M <= 16), beside the
// token-stream forward: T [M, r] (fp32, saved for the backward) and
// bf16(s*T) [M, rp] (the low-rank activations the forward's last step uses).
//
// Operation: the LoRA_A product of the fused chain Linear -> LoRA_A -> LoRA_B ->
// Add ("UnSloth加速原理：CUDA内核融合与内存优化", section "内核融合").  With so few
// tokens this is a read of A (d_in x r) and little else, so it runs as one
// thread-block cluster of eight CTAs beside the weight stream:
//   * CTA k of the cluster takes the k-th eighth of the contraction (in steps
//     of 16 input features).  Its rows of A are contiguous in memory, so they
//     come in by bulk copies of 32 KB chunks (with the matching columns of X)
//     through a ring of three shared-memory buffers: few, long DRAM reads.
//   * The four warps take alternate steps of each chunk and accumulate with
//     mma.sync (X rows as the A operand, columns of A as the B operand,
//     bf16 -> fp32); the warps are added in shared memory, and each CTA adds
//     the eight CTAs' sums, in rank order, for its eighth of T's elements
//     through distributed shared memory -- a fixed order, so T does not
//     depend on timing.
// Every mbarrier wait is bounded (kWaitLimitNs): on expiry the CTA records a
// timeout in the status word and winds down.

#include <cuda_bf16.h>
#include <algorithm>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace qlora {
namespace {

constexpr int kCluster = 8;
constexpr int kXaWarps = 4;
constexpr int kXaThreads = kXaWarps * 32;
constexpr int kBufs = 3;                     // chunks in flight
constexpr int kChunkA = 32 * 1024;           // bytes of A per chunk
constexpr int kMaxChunkSteps = 32;          // 16-feature steps per chunk at most (512 features)
constexpr int kXChunkPitch = kMaxChunkSteps * 16 * 2 + 16;   // bytes per token row of a chunk's X columns

template <int RP>
struct XaSmem {
  static constexpr int kAOff = 0;
  static constexpr int kXOff = kBufs * kChunkA;
  static constexpr int kRedOff = kXOff + kBufs * 16 * kXChunkPitch;
  static constexpr int kCsumOff = kRedOff + kXaWarps * 16 * RP * 4;
  static constexpr int kBarOff = kCsumOff + 16 * RP * 4;
  static constexpr int kBytes = kBarOff + 8 * kBufs + 16;
  static_assert(kBytes <= 227 * 1024, "fits the shared memory of one CTA");
};

struct XaParams {
  const uint16_t* X;     // [M, K] bf16
  const uint16_t* A;     // [K, a_cols] bf16 (a_cols = r, or rp for the zero-padded copy)
  float* T;              // [M, r] fp32
  uint16_t* s_t;         // [M, rp] bf16(s*T)
  int* status;
  int M, K, r, rp, a_cols;
  float s;
};

__device__ __forceinline__ void mma_16816_xa(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32_xa(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// RP = rp (64 or 128): the columns of T computed, 8 per MMA.
template <int RP>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kXaThreads, 1)
    lora_xa_small_kernel(const XaParams p) {
  using S = XaSmem<RP>;
  constexpr int JG = RP / 8;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  const uint32_t base = (smem_u32(smem_raw) + 15u) & ~15u;
  uint8_t* const gbase = smem_raw + (base - smem_u32(smem_raw));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g4 = lane >> 2, t = lane & 3;
  const uint32_t rank = cluster_ctarank();
  auto bar = [&](int b) { return base + S::kBarOff + 8u * b; };
  Abort ab{&s_abort, p.status};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int b = 0; b < kBufs; ++b) mbar_init(bar(b), 1);
    fence_barrier_init();
  }
  // X rows of tokens past M are zero
  for (int i = threadIdx.x; i < kBufs * 16 * (kXChunkPitch / 16); i += kXaThreads)
    if ((i / (kXChunkPitch / 16)) % 16 >= p.M)
      st_shared_v4(base + S::kXOff + static_cast<uint32_t>(i) * 16u, make_uint4(0u, 0u, 0u, 0u));
  __syncthreads();
  // launched with programmatic serialisation, this first kernel of the call may
  // start while the previous kernel on the stream runs: the set-up above
  // overlaps it; global memory is touched only after it has completed.  Then
  // the token-stream kernel may be scheduled (it reads the call's inputs at
  // once, and waits for this grid before its end, for T).
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();

  // this CTA's steps of the contraction, in chunks
  const int steps = p.K / 16;
  const int st0 = static_cast<int>(static_cast<int64_t>(steps) * rank / kCluster);
  const int st1 = static_cast<int>(static_cast<int64_t>(steps) * (rank + 1) / kCluster);
  // steps per chunk: as many as 32 KB of A's rows hold, at most 32
  const int chunk_steps = min(kMaxChunkSteps, kChunkA / (16 * 2 * p.a_cols));
  const int n_chunks = (st1 - st0 + chunk_steps - 1) / chunk_steps;
  auto issue = [&](int c) {
    const int b = c % kBufs;
    const int c0 = st0 + c * chunk_steps, c1 = min(st1, c0 + chunk_steps);
    const uint32_t a_bytes = static_cast<uint32_t>((c1 - c0) * 16 * p.a_cols * 2);
    const uint32_t x_bytes = static_cast<uint32_t>((c1 - c0) * 16 * 2);
    mbar_arrive_expect_tx(bar(b), a_bytes + x_bytes * static_cast<uint32_t>(p.M));
    bulk_load_1d(base + S::kAOff + static_cast<uint32_t>(b * kChunkA), p.A + static_cast<int64_t>(c0) * 16 * p.a_cols,
                 a_bytes, bar(b));
    for (int tok = 0; tok < p.M; ++tok)
      bulk_load_1d(base + S::kXOff + static_cast<uint32_t>((b * 16 + tok) * kXChunkPitch),
                   p.X + static_cast<int64_t>(tok) * p.K + c0 * 16, x_bytes, bar(b));
  };
  if (threadIdx.x == 0)
    for (int c = 0; c < kBufs && c < n_chunks; ++c) issue(c);

  float acc[JG][4];
#pragma unroll
  for (int jg = 0; jg < JG; ++jg) acc[jg][0] = acc[jg][1] = acc[jg][2] = acc[jg][3] = 0.0f;
  bool ok = true;
  int c = 0;
  for (; c < n_chunks; ++c) {
    const int b = c % kBufs;
    if (!__syncthreads_and(mbar_wait_spin(bar(b), (c / kBufs) & 1, ab))) {
      ok = false;
      break;
    }
    const int c0 = st0 + c * chunk_steps, c1 = min(st1, c0 + chunk_steps);
    const uint32_t a_buf = base + S::kAOff + static_cast<uint32_t>(b * kChunkA);
    const uint32_t x_a = base + S::kXOff + static_cast<uint32_t>((b * 16 + g4) * kXChunkPitch);
    const uint32_t x_b = x_a + 8u * kXChunkPitch;
    for (int ks = warp; ks < c1 - c0; ks += kXaWarps) {
      const uint32_t k0 = static_cast<uint32_t>(16 * ks + 2 * t);
      // X as the A operand: rows g, g+8 (tokens), columns k0, k0+1 and k0+8, k0+9
      const uint32_t a[4] = {lds32_xa(x_a + k0 * 2u), lds32_xa(x_b + k0 * 2u),
                             lds32_xa(x_a + (k0 + 8u) * 2u), lds32_xa(x_b + (k0 + 8u) * 2u)};
      const uint32_t row = a_buf + k0 * static_cast<uint32_t>(p.a_cols) * 2u;
#pragma unroll
      for (int jg = 0; jg < JG; ++jg) {
        // A as the B operand: column j = 8 jg + g, rows k0, k0+1 and k0+8, k0+9
        const int j = 8 * jg + g4;
        uint32_t b0 = 0u, b1 = 0u;
        if (j < p.a_cols) {
          const uint32_t at = row + static_cast<uint32_t>(j) * 2u, pitch = static_cast<uint32_t>(p.a_cols) * 2u;
          b0 = lds_u16(at) | (lds_u16(at + pitch) << 16);
          b1 = lds_u16(at + 8u * pitch) | (lds_u16(at + 9u * pitch) << 16);
        }
        mma_16816_xa(acc[jg], a, b0, b1);
      }
    }
    // every warp is done with buffer b: refill it
    __syncthreads();
    if (threadIdx.x == 0 && c + kBufs < n_chunks) {
      fence_proxy_async_smem();
      issue(c + kBufs);
    }
  }
  if (!ok) {
    // a wait ran out: let the copies issued land, then leave with the cluster
    if (threadIdx.x == 0)
      for (int q = c; q < n_chunks && q < c + kBufs; ++q) mbar_wait_spin(bar(q % kBufs), (q / kBufs) & 1, ab, false);
  }
  // c0, c1: token g, columns 8 jg + 2t, +1; c2, c3: token g + 8
  float* const red = reinterpret_cast<float*>(gbase + S::kRedOff) + warp * 16 * RP;
#pragma unroll
  for (int jg = 0; jg < JG; ++jg) {
    red[g4 * RP + 8 * jg + 2 * t] = acc[jg][0];
    red[g4 * RP + 8 * jg + 2 * t + 1] = acc[jg][1];
    red[(g4 + 8) * RP + 8 * jg + 2 * t] = acc[jg][2];
    red[(g4 + 8) * RP + 8 * jg + 2 * t + 1] = acc[jg][3];
  }
  __syncthreads();
  const float* const red0 = reinterpret_cast<const float*>(gbase + S::kRedOff);
  float* const csum = reinterpret_cast<float*>(gbase + S::kCsumOff);
  for (int e = threadIdx.x; e < 16 * RP; e += kXaThreads) {
    float v = red0[e];
#pragma unroll
    for (int q = 1; q < kXaWarps; ++q) v += red0[q * 16 * RP + e];
    csum[e] = v;
  }
  // every CTA's sum is in shared memory after this barrier
  cluster_sync_all();
  {
    // CTA k adds the eight sums, in rank order, for every eighth element
    const uint32_t local = base + S::kCsumOff;
    for (int e = static_cast<int>(rank) + kCluster * threadIdx.x; e < p.M * RP; e += kCluster * kXaThreads) {
      const int tok = e / RP, j = e % RP;
      const uint32_t off = static_cast<uint32_t>(e) * 4u;
      float part[kCluster];
#pragma unroll
      for (int q = 0; q < kCluster; ++q) part[q] = ld_dsmem_f32(map_to_cta(local + off, q));
      float v = part[0];
#pragma unroll
      for (int q = 1; q < kCluster; ++q) v += part[q];
      if (j < p.r) p.T[static_cast<int64_t>(tok) * p.r + j] = v;
      p.s_t[static_cast<int64_t>(tok) * p.rp + j] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(p.s, v)));
    }
  }
  // nobody leaves while a peer may still read its shared memory
  cluster_sync_all();
}

template <int RP>
cudaError_t launch_xa_rp(const XaParams& p, cudaStream_t stream) {
  auto kern = lora_xa_small_kernel<RP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, XaSmem<RP>::kBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster, 1, 1);
  cfg.blockDim = dim3(kXaThreads, 1, 1);
  cfg.dynamicSmemBytes = XaSmem<RP>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchScope scope(kKindRowsT, stream);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

cudaError_t launch_xa_small(const LayerDims& d, const uint16_t* X, const uint16_t* A, int a_cols, float* XA,
                            const Workspace& ws, int* status, cudaStream_t stream) {
  XaParams p;
  p.X = X;
  p.A = A;
  p.T = XA;
  p.s_t = ws.s_t;
  p.status = status;
  p.M = d.M;
  p.K = d.K;
  p.r = d.r;
  p.rp = d.rp;
  p.a_cols = a_cols;
  p.s = d.s;
  if (d.rp == 64) return launch_xa_rp<64>(p, stream);
  return launch_xa_rp<128>(p, stream);
}

}  // namespace qlora
