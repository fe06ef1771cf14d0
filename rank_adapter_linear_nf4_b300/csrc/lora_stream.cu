// lora_stream.cu -- the forward Y = X . W_deq^T + s . (X . A) . B for a handful of
// tokens (M <= 16), where the layer is a stream of its NF4 weight.
//
// Operation: the fused QLoRA linear of the Unsloth pages ("UnSloth加速原理：CUDA内核
// 融合与内存优化", section "内核融合"; "这不是“魔法”是把Unsloth的底层优化逻辑榨干了用",
// section 1), the same result as the main kernel.  With so few tokens the work is
// 0.5625 bytes of codes and absmax per weight element against 2*M flops, so the
// kernel is built around keeping enough of the weight in flight to run at the
// HBM rate, with nothing that makes a warp wait for another:
//
//   * Work item: 32 weight rows (two 16-row MMA groups) x one 64-element NF4
//     block.  Items are numbered row-pair-major (all blocks of rows 0..31, then
//     rows 32..63, ...) and every warp of a persistent grid (one CTA per SM)
//     takes an equal contiguous range of them.
//   * Each lane loads its quarter of each block row (8 code bytes = 16
//     elements) for four rows straight into registers with 8-byte loads that
//     skip L1, several items ahead of the one it computes (a ring of
//     registers): no shared-memory staging, no barriers.  X comes through L1
//     with 16-byte loads (every warp of the SM reads the same X).
//   * Decode: one shared-memory lookup per code byte in a table of the 256
//     possible bytes -> a pair of bf16 levels, one copy per lane (32 KB, never a
//     bank conflict), straight into the A registers of mma.sync m16n8k16
//     (bf16 -> fp32).  The block's absmax multiplies the block's MMA sum in
//     fp32: the sum of bf16(level[q]) * x * absmax, which is the sum of
//     bf16(level[q] * absmax) * x up to the rounding of the weight (both are
//     within 2^-9 of level[q] * absmax).
//   * The contraction order inside an MMA is free: lane (g, t) of the MMA
//     takes elements 16t .. 16t+15 of the block (its 8 code bytes; k-step s
//     uses bytes 2s and 2s+1), and the X fragments are read in that order.
//   * Where a warp's range crosses into the next row pair it writes the
//     finished segment's fp32 partial to its own slot in the workspace.  After
//     its range, the warp counts its segments in per-row-pair counters; the
//     warp that completes a row pair's count adds the pair's partials in warp
//     order (so results do not depend on timing), adds the low-rank term
//     bf16(s*T) . B with mma.sync, and stores the 32 rows of Y.
//   * bf16(s*T) and the zeroed counters come from the rank-r kernel launched
//     before this one; this kernel is launched with programmatic serialisation
//     and waits for that kernel (griddepcontrol.wait) only after its stream.
//
// No wait in this kernel depends on another CTA: the reduction is by atomic
// counters and the last warp to arrive, so there is nothing that can hang.

#include <cuda_bf16.h>
#include <cstdint>
#include <algorithm>
#include <cstring>

#include "kernels.h"
#include "nf4_lut.cuh"
#include "ptx.cuh"

namespace qlora {
namespace {

constexpr int kWarps = 16;                   // warps per CTA (one CTA per SM)
constexpr int kThreads = kWarps * 32;
constexpr int kPairRows = 32;                // weight rows per item
constexpr int kRing = 4;                     // items whose codes are in flight per warp
constexpr int kLutWords = 256 * 32;          // 256 code bytes x 32 lane copies
constexpr int kMinItemsPerWarp = 4;

// bf16 bit patterns (round to nearest even) of the NF4 levels, in code order:
// the host copy kNF4LevelsHost rounded; launch_stream_fwd checks the two agree.
constexpr uint16_t kLevelBf16[16] = {0xBF80, 0xBF32, 0xBF06, 0xBECA, 0xBE92, 0xBE3D, 0xBDBA, 0x0000,
                                     0x3DA3, 0x3E25, 0x3E7C, 0x3EAD, 0x3EE2, 0x3F10, 0x3F39, 0x3F80};
__constant__ uint16_t c_level_bf16[16] = {0xBF80, 0xBF32, 0xBF06, 0xBECA, 0xBE92, 0xBE3D, 0xBDBA, 0x0000,
                                          0x3DA3, 0x3E25, 0x3E7C, 0x3EAD, 0x3EE2, 0x3F10, 0x3F39, 0x3F80};

struct StreamParams {
  const uint16_t* X;        // [M, K] bf16
  const uint8_t* codes;     // [N, K/2]
  const float* absmax;      // [N, K/64]
  const uint16_t* B;        // [r, N] bf16
  const uint16_t* s_t;      // [M, rp] bf16(s*T), zero columns r..rp-1
  uint16_t* Y;              // [M, N] bf16
  float* partials;          // slots of 256 * MT floats, slot = global warp + row pair
  int* counters;            // [row pairs], zero at launch
  int M, K, N, r, rp;
  int kb;                   // NF4 blocks per row: K / 64
  int pairs;                // row pairs: ceil(N / 32)
  long long items;          // pairs * kb
  long long warps;          // warps with work: min(items, warps of the grid); each takes >= 1 item
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// 8 bytes of codes, streamed once: no L1 allocation.
__device__ __forceinline__ uint2 ldg_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ldg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// D += A . B for one m16n8k16 tile, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The pair-table word of code byte `sel & 3` of w, from this lane's copy
// (entry v of lane l at byte offset 128 v + 4 l; lut_lane = table + 4 l).
__device__ __forceinline__ uint32_t lut_pair(uint32_t lut_lane, uint32_t w, uint32_t sel) {
  return lds32(prmt(w, 0u, sel) * 128u + lut_lane);
}

// One item's weight loads: rows g, g+8, g+16, g+24 of the pair (g = lane / 4),
// bytes 8t .. 8t+7 of the block (t = lane % 4), and the four rows' absmax.
struct ItemLoad {
  uint2 code[4];
  float am[4];
};

__device__ __forceinline__ void load_item(ItemLoad& it, const StreamParams& p, int pair, int b, int g4, int t) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int n = pair * kPairRows + g4 + 8 * q;
    const int nc = n < p.N ? n : p.N - 1;   // rows past the weight: any row, weight 0 below
    it.code[q] = ldg_stream_v2(p.codes + static_cast<int64_t>(nc) * (p.K >> 1) + b * 32 + t * 8);
    const float a = ldg_nc_f32(p.absmax + static_cast<int64_t>(nc) * p.kb + b);
    it.am[q] = n < p.N ? a : 0.0f;
  }
}

// X fragments of block b: token half j (tokens 8j + g), elements 16t .. 16t+15.
template <int MT>
__device__ __forceinline__ void load_x(uint4 (&x)[MT][2], const StreamParams& p, int b, int g4, int t) {
#pragma unroll
  for (int j = 0; j < MT; ++j) {
    const int tok = min(8 * j + g4, p.M - 1);   // tokens past M: any row; their outputs are never stored
    const uint16_t* src = p.X + static_cast<int64_t>(tok) * p.K + b * 64 + t * 16;
    x[j][0] = ldg_v4(src);
    x[j][1] = ldg_v4(src + 8);
  }
}

// acc[h] += absmax * (this item's MMA sum) for the two 16-row groups h.
template <int MT>
__device__ __forceinline__ void compute_item(const ItemLoad& it, const uint4 (&x)[MT][2], uint32_t lut_lane,
                                             float (&acc)[2][MT][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint2 ca = it.code[2 * h], cb = it.code[2 * h + 1];   // rows g (+16h) and g+8 (+16h)
    float d[MT][4];
#pragma unroll
    for (int j = 0; j < MT; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.0f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      // k-step s: code bytes 2s (fragment columns 2t, 2t+1) and 2s+1 (2t+8, 2t+9)
      const uint32_t wa = s < 2 ? ca.x : ca.y, wb = s < 2 ? cb.x : cb.y;
      const uint32_t sel0 = 0x4440u | static_cast<uint32_t>((2 * s) & 3);
      const uint32_t sel1 = 0x4440u | static_cast<uint32_t>((2 * s + 1) & 3);
      const uint32_t a[4] = {lut_pair(lut_lane, wa, sel0), lut_pair(lut_lane, wb, sel0),
                             lut_pair(lut_lane, wa, sel1), lut_pair(lut_lane, wb, sel1)};
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const uint32_t b0 = (s & 1) ? (s < 2 ? x[j][0].z : x[j][1].z) : (s < 2 ? x[j][0].x : x[j][1].x);
        const uint32_t b1 = (s & 1) ? (s < 2 ? x[j][0].w : x[j][1].w) : (s < 2 ? x[j][0].y : x[j][1].y);
        mma_16816(d[j], a, b0, b1);
      }
    }
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      acc[h][j][0] = fmaf(it.am[2 * h], d[j][0], acc[h][j][0]);
      acc[h][j][1] = fmaf(it.am[2 * h], d[j][1], acc[h][j][1]);
      acc[h][j][2] = fmaf(it.am[2 * h + 1], d[j][2], acc[h][j][2]);
      acc[h][j][3] = fmaf(it.am[2 * h + 1], d[j][3], acc[h][j][3]);
    }
  }
}

// The warp whose range holds item x (ranges are [items*w/W, items*(w+1)/W)).
__device__ __forceinline__ long long owner_warp(long long x, long long items, long long W) {
  return ((x + 1) * W - 1) / items;
}

template <int MT>
__device__ __forceinline__ float* slot_ptr(const StreamParams& p, long long slot, int lane) {
  return p.partials + slot * (256 * MT) + lane * 4;
}

template <int MT>
__device__ __forceinline__ void store_partial(const StreamParams& p, long long slot, int lane,
                                              const float (&acc)[2][MT][4]) {
  float* dst = slot_ptr<MT>(p, slot, lane);
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int j = 0; j < MT; ++j)
      __stcg(reinterpret_cast<float4*>(dst + (h * MT + j) * 128),
             make_float4(acc[h][j][0], acc[h][j][1], acc[h][j][2], acc[h][j][3]));
}

// Finishes row pair `pair`: its partials in warp order, the low-rank term, Y.
template <int MT>
__device__ __forceinline__ void finish_pair(const StreamParams& p, int pair, long long W, int lane) {
  const int g4 = lane >> 2, t = lane & 3;
  const long long first = owner_warp(static_cast<long long>(pair) * p.kb, p.items, W);
  const long long last = owner_warp(static_cast<long long>(pair) * p.kb + p.kb - 1, p.items, W);
  float acc[2][MT][4];
  {
    const float* src = slot_ptr<MT>(p, first + pair, lane);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (h * MT + j) * 128));
        acc[h][j][0] = v.x;
        acc[h][j][1] = v.y;
        acc[h][j][2] = v.z;
        acc[h][j][3] = v.w;
      }
  }
  for (long long w = first + 1; w <= last; ++w) {
    const float* src = slot_ptr<MT>(p, w + pair, lane);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (h * MT + j) * 128));
        acc[h][j][0] += v.x;
        acc[h][j][1] += v.y;
        acc[h][j][2] += v.z;
        acc[h][j][3] += v.w;
      }
  }
  // low-rank term: D += B^T (rows n, columns j) . bf16(s*T)^T (rows j, columns tokens)
  const uint16_t* Bp = p.B;
  for (int j0 = 0; j0 < p.rp; j0 += 16) {
    uint32_t bt[MT][2];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      const int tok = 8 * j + g4;
      const uint32_t* row = reinterpret_cast<const uint32_t*>(p.s_t + static_cast<int64_t>(tok < p.M ? tok : 0) * p.rp);
      bt[j][0] = tok < p.M ? __ldcg(row + ((j0 + 2 * t) >> 1)) : 0u;
      bt[j][1] = tok < p.M ? __ldcg(row + ((j0 + 2 * t + 8) >> 1)) : 0u;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int na = pair * kPairRows + 16 * h + g4, nb = na + 8;
      auto bval = [&](int jj, int n) -> uint32_t {
        return (jj < p.r && n < p.N) ? static_cast<uint32_t>(__ldg(Bp + static_cast<int64_t>(jj) * p.N + n)) : 0u;
      };
      const int ja = j0 + 2 * t;
      const uint32_t a[4] = {bval(ja, na) | (bval(ja + 1, na) << 16), bval(ja, nb) | (bval(ja + 1, nb) << 16),
                             bval(ja + 8, na) | (bval(ja + 9, na) << 16), bval(ja + 8, nb) | (bval(ja + 9, nb) << 16)};
#pragma unroll
      for (int j = 0; j < MT; ++j) mma_16816(acc[h][j], a, bt[j][0], bt[j][1]);
    }
  }
  // Y: c0, c1 -> row g (+16h), tokens 2t, 2t+1; c2, c3 -> row g+8
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int na = pair * kPairRows + 16 * h + g4, nb = na + 8;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      const int tok = 8 * j + 2 * t;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int n = (e < 2) ? na : nb, tk = tok + (e & 1);
        if (n < p.N && tk < p.M)
          p.Y[static_cast<int64_t>(tk) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[h][j][e]));
      }
    }
  }
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1) lora_stream_kernel(const StreamParams p) {
  __shared__ __align__(16) uint32_t s_lut[kLutWords];
  // the decode table: word 32 v + l holds bf16(level[v >> 4]) (the byte's first
  // element) in its low half and bf16(level[v & 15]) in its high half
  for (int i = threadIdx.x; i < kLutWords; i += kThreads) {
    const int v = i >> 5;
    s_lut[i] = static_cast<uint32_t>(c_level_bf16[v >> 4]) | (static_cast<uint32_t>(c_level_bf16[v & 15]) << 16);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g4 = lane >> 2, t = lane & 3;
  const uint32_t lut_lane = smem_u32(s_lut) + static_cast<uint32_t>(lane) * 4u;
  const long long W = p.warps;
  const long long wg = static_cast<long long>(blockIdx.x) * kWarps + warp;
  const long long lo = wg < W ? p.items * wg / W : 0, hi = wg < W ? p.items * (wg + 1) / W : 0;

  if (lo < hi) {
    // ring of code loads, kRing items ahead
    ItemLoad ring[kRing];
    int lpair = static_cast<int>(lo / p.kb), lb = static_cast<int>(lo % p.kb);   // next item to load
#pragma unroll
    for (int u = 0; u < kRing; ++u) {
      if (lo + u < hi) load_item(ring[u], p, lpair, lb, g4, t);
      if (++lb == p.kb) {
        lb = 0;
        ++lpair;
      }
    }
    int cpair = static_cast<int>(lo / p.kb), cb = static_cast<int>(lo % p.kb);   // item being computed
    uint4 xn[MT][2];
    load_x<MT>(xn, p, cb, g4, t);
    float acc[2][MT][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < MT; ++j) acc[h][j][0] = acc[h][j][1] = acc[h][j][2] = acc[h][j][3] = 0.0f;

    for (long long base = lo; base < hi; base += kRing) {
#pragma unroll
      for (int u = 0; u < kRing; ++u) {
        const long long i = base + u;
        if (i < hi) {
          uint4 x[MT][2];
#pragma unroll
          for (int j = 0; j < MT; ++j) {
            x[j][0] = xn[j][0];
            x[j][1] = xn[j][1];
          }
          // the next item's X, one item ahead (it is an L1 hit most of the time)
          const int nb = cb + 1 == p.kb ? 0 : cb + 1;
          if (i + 1 < hi) load_x<MT>(xn, p, nb, g4, t);
          compute_item<MT>(ring[u], x, lut_lane, acc);
          // refill this ring slot kRing items ahead
          if (i + kRing < hi) load_item(ring[u], p, lpair, lb, g4, t);
          if (++lb == p.kb) {
            lb = 0;
            ++lpair;
          }
          // end of a row pair's segment, or of the range: park the partial
          const bool seg_end = (nb == 0) || (i + 1 == hi);
          if (seg_end) {
            store_partial<MT>(p, wg + cpair, lane, acc);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int j = 0; j < MT; ++j) acc[h][j][0] = acc[h][j][1] = acc[h][j][2] = acc[h][j][3] = 0.0f;
          }
          cb = nb;
          if (nb == 0) ++cpair;
        }
      }
    }
  }

  // bf16(s*T) and the zeroed counters come from the kernel before this one
  griddep_wait();
  if (lo >= hi) return;
  __threadfence();   // this lane's partial stores, before the warp's counter updates
  __syncwarp();
  const int pair_first = static_cast<int>(lo / p.kb), pair_last = static_cast<int>((hi - 1) / p.kb);
  for (int pair = pair_first; pair <= pair_last; ++pair) {
    const long long first = owner_warp(static_cast<long long>(pair) * p.kb, p.items, W);
    const long long last = owner_warp(static_cast<long long>(pair) * p.kb + p.kb - 1, p.items, W);
    int arrived = 0;
    if (lane == 0) arrived = atomicAdd(p.counters + pair, 1);
    arrived = __shfl_sync(0xffffffffu, arrived, 0);
    if (arrived == static_cast<int>(last - first)) {
      __threadfence();   // the other warps' partials, after their counter updates
      finish_pair<MT>(p, pair, W, lane);
    }
  }
}

template <int MT>
cudaError_t launch_stream_mt(const StreamParams& p, int grid, cudaStream_t stream) {
  auto kern = lora_stream_kernel<MT>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // programmatic serialisation: the weight stream starts while the rank-r
  // kernel before this one finishes; bf16(s*T) and the counters wait for it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchScope scope(kKindStream, stream);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

long long stream_items(const LayerDims& d) {
  return static_cast<long long>((d.N + kPairRows - 1) / kPairRows) * (d.K / 64);
}

int stream_grid(const LayerDims& d, int sms) {
  const long long want = (stream_items(d) + kWarps * kMinItemsPerWarp - 1) / (kWarps * kMinItemsPerWarp);
  return static_cast<int>(want < sms ? (want < 1 ? 1 : want) : sms);
}

}  // namespace

int stream_counter_slots(const LayerDims& d) { return (d.N + kPairRows - 1) / kPairRows; }

size_t stream_partial_bytes(const LayerDims& d, int sms) {
  const int mt = d.M <= 8 ? 1 : 2;
  const long long slots = static_cast<long long>(stream_grid(d, sms)) * kWarps + stream_counter_slots(d);
  return static_cast<size_t>(slots) * 256 * mt * sizeof(float);
}

bool stream_applies(const LayerDims& d, const Workspace& ws, int sms) {
  if (d.M < 1 || d.M > kStreamMaxTokens || d.K % 64 != 0) return false;
  if (ws.counters == nullptr || ws.partials == nullptr || ws.counter_cap < stream_counter_slots(d)) return false;
  return ws.partial_bytes >= stream_partial_bytes(d, sms);
}

// The compile-time bf16 table against the fp32 levels, rounded to nearest even.
bool level_table_matches() {
  for (int i = 0; i < 16; ++i) {
    uint32_t u;
    std::memcpy(&u, &kNF4LevelsHost[i], sizeof(u));
    const uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    if (r != kLevelBf16[i]) return false;
  }
  return true;
}

cudaError_t launch_stream_fwd(const LayerDims& d, const uint16_t* X, const uint8_t* packed, const float* absmax,
                              const uint16_t* B, const Workspace& ws, uint16_t* Y, int* status, int sms,
                              cudaStream_t stream) {
  (void)status;   // nothing in this kernel waits, so nothing can time out
  static const bool table_ok = level_table_matches();
  if (!table_ok) return cudaErrorInvalidValue;
  StreamParams p;
  p.X = X;
  p.codes = packed;
  p.absmax = absmax;
  p.B = B;
  p.s_t = ws.s_t;
  p.Y = Y;
  p.partials = ws.partials;
  p.counters = ws.counters;
  p.M = d.M;
  p.K = d.K;
  p.N = d.N;
  p.r = d.r;
  p.rp = d.rp;
  p.kb = d.K / 64;
  p.pairs = stream_counter_slots(d);
  p.items = stream_items(d);
  const int grid = stream_grid(d, sms);
  p.warps = std::min<long long>(p.items, static_cast<long long>(grid) * kWarps);
  if (d.M <= 8) return launch_stream_mt<1>(p, grid, stream);
  return launch_stream_mt<2>(p, grid, stream);
}

}  // namespace qlora
