// lora_kernels.cu -- the fused NF4-QLoRA linear layer on sm_103a.
//
// Forward  Y  = X . W_deq^T + s . (X . A) . B
// Backward dX = dY . W_deq + s . (dY . B^T) . A^T,  dA = s . X^T . G,  dB = s . T^T . dY
// (Unsloth pages: "UnSloth加速原理：CUDA内核融合与内存优化", section "内核融合" for the fused
// Linear + LoRA + add chain; "Unsloth性能实测：比传统方法快2倍真的吗？", section 3.2 for
// the hand-written backward.)
//
// Kernels:
//  * lora_prep_kernel   -- pads A to [K, rp], transposes B to [N, rp], and (backward)
//                          turns the saved fp32 T into bf16(s*T) [M, rp].
//  * lora_skinny_kernel -- the rank-r contractions on the tensor core:
//        rows  T = X.A  (also writes bf16(s*T)),  G-side bf16(s * dY.B^T)
//        red   dA = X^T . bf16(s*G),  dB = (bf16(s*T))^T . dY
//      one 128-row tile per CTA; the contraction is split over the CTAs of a
//      thread-block cluster and the partial tiles are summed in a fixed order
//      through distributed shared memory (deterministic, no atomics).
//  * lora_main_kernel   -- the dominant GEMM.  Output features (rows of W for Y,
//      columns of W for dX) are the UMMA M dimension (128 per CTA) and tokens
//      the N dimension (up to 256).  Dequantising warps expand NF4 blocks
//      straight into the 128-byte-swizzled shared-memory operand the tensor
//      core reads (K-major for Y, MN-major for dX, where W is used
//      transposed); TMA brings the token tiles; the LoRA term is one or two
//      extra 64-wide K stages ([bf16(s*T) | ...] against B^T, or bf16(s*G)
//      against A) accumulated into the same TMEM tile; the epilogue converts
//      TMEM to bf16 and writes the tile with a TMA store.
#include <algorithm>
#include <cstdio>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "nf4_lut.cuh"
#include "ptx.cuh"

namespace qlora {

namespace {

constexpr int kTileP = 128;   // UMMA M: output features (main) / output rows (skinny)
constexpr int kTileK = 64;    // contraction elements per stage (one 128-B swizzle row)

// ============================================================== prep

// Zero-padded copy of A, [K, rp], for ranks whose rows are not 16-byte
// multiples (the TMA reads rows of 16-byte multiples).
struct PrepParams {
  const uint16_t* A;      // [K, r]
  uint16_t* a_pad;        // [K, rp]
  int64_t n_apad;
  int N, r, rp;
  float s;
};

__global__ void __launch_bounds__(256) lora_prep_kernel(const PrepParams p) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < p.n_apad;
       e += stride) {
    const int64_t k = e / p.rp;
    const int j = static_cast<int>(e - k * p.rp);
    p.a_pad[e] = (j < p.r) ? p.A[k * p.r + j] : uint16_t(0);
  }
}

// ============================================================== skinny (rank-r) contractions

// kRowsT: T = X . A          A operand X tile (K-major), B operand A (MN-major); writes T and bf16(s*T)
// kRowsG: G = dY . B^T       A operand dY tile (K-major), B operand B (K-major); writes bf16(s*G) and,
//                            for the same rows, bf16(s*T) from the saved fp32 T
// kRed:   job 0  dA = X^T . bf16(s*G)    job 1  dB = (bf16(s*T))^T . dY   (both operands MN-major)
enum SkinnyMode : int { kRowsT = 0, kRowsG = 1, kRed = 2 };

constexpr int kSkStages = 6;
constexpr int kSkThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue

template <int RP>
struct SkinnySmem {
  static constexpr int kABytes = kTileP * 128;   // 128 rows x 64 bf16
  static constexpr int kBBytes = RP * 128;       // RP columns x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = kSkStages * kStageBytes;
  static constexpr int kBytes = kBarOffset + 256 + 1024;
  static constexpr int kRedStride = RP + 4;      // floats per reduction row: 16-B rows, spread banks
  static_assert(kTileP * kRedStride * 4 <= kBarOffset, "reduction buffer must fit");
};

struct SkinnyJob {
  int rows;            // extent of the output row dimension
  int tiles;           // 128-row tiles of this job
  float* out_f32;      // kRowsT: T [rows, r]; kRed job 0: dA [rows, r]; kRed job 1: dB [r, rows]
  uint16_t* out_bf16;  // kRowsT: bf16(s*T) [rows, RP]; kRowsG: bf16(s*G) [rows, RP]
};

struct SkinnyParams {
  int r;               // LoRA rank (valid output columns)
  int num_ct;          // contraction tiles of 64
  float s;             // scale for the rows modes
  SkinnyJob job[2];    // kRed: job 0 = dA, job 1 = dB; the rows modes use job 0
  const float* xa;     // kRowsG: saved T [rows, r]
  uint16_t* s_t;       // kRowsG: bf16(s*T) [rows, RP] written from xa
  int* status;
};

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(cluster_addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ uint2 bf16x4_scaled(float s, float4 v) {
  uint2 o;
  o.x = pack_bf16x2(__fmul_rn(s, v.x), __fmul_rn(s, v.y));
  o.y = pack_bf16x2(__fmul_rn(s, v.z), __fmul_rn(s, v.w));
  return o;
}

template <int MODE, int RP>
__global__ void __launch_bounds__(kSkThreads, 1)
    lora_skinny_kernel(const __grid_constant__ CUtensorMap map_a0,
                       const __grid_constant__ CUtensorMap map_b0,
                       const __grid_constant__ CUtensorMap map_a1,
                       const __grid_constant__ CUtensorMap map_b1, const SkinnyParams p) {
  constexpr bool kAmn = (MODE == kRed);      // A operand MN-major
  constexpr bool kBmn = (MODE != kRowsG);    // B operand MN-major
  using S = SkinnySmem<RP>;

  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t bar0 = base + S::kBarOffset;
  const uint32_t accum_bar = bar0 + 8u * (2 * kSkStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int job = (MODE == kRed && static_cast<int>(blockIdx.x) >= p.job[0].tiles) ? 1 : 0;
  // job fields picked with selects (a dynamic index into the parameter struct would spill it)
  const int j_rows = job ? p.job[1].rows : p.job[0].rows;
  float* const j_out_f32 = job ? p.job[1].out_f32 : p.job[0].out_f32;
  uint16_t* const j_out_bf16 = p.job[0].out_bf16;
  const CUtensorMap* map_a = job ? &map_a1 : &map_a0;
  const CUtensorMap* map_b = job ? &map_b1 : &map_b0;
  const int p0 = (static_cast<int>(blockIdx.x) - (job ? p.job[0].tiles : 0)) * kTileP;
  const uint32_t nsplit = gridDim.y;
  const uint32_t split = blockIdx.y;
  const int ct_begin = static_cast<int>((static_cast<int64_t>(p.num_ct) * split) / nsplit);
  const int ct_end = static_cast<int>((static_cast<int64_t>(p.num_ct) * (split + 1)) / nsplit);
  const int nct = ct_end - ct_begin;
  Abort ab{&s_abort, p.status};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kSkStages; ++i) {
      mbar_init(bar0 + 8u * i, 1);                    // full
      mbar_init(bar0 + 8u * (kSkStages + i), 1);      // empty
    }
    mbar_init(accum_bar, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(map_a);
    tma_prefetch_map(map_b);
  }
  if (warp == 1) tmem_alloc(smem_u32(&s_tmem), RP);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_d = s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      int i = 0;
      for (; i < nct; ++i) {
        const int slot = i % kSkStages;
        const uint32_t ph = (i / kSkStages) & 1;
        if (!mbar_wait(bar0 + 8u * (kSkStages + slot), ph ^ 1, ab)) break;
        const int ct = ct_begin + i;
        const uint32_t a = base + slot * S::kStageBytes;
        const uint32_t b = a + S::kABytes;
        const uint32_t full = bar0 + 8u * slot;
        mbar_arrive_expect_tx(full, S::kStageBytes);
        if (kAmn) {
          tma_load_2d(a, map_a, full, p0, ct * kTileK);
          tma_load_2d(a + 8192, map_a, full, p0 + 64, ct * kTileK);
        } else {
          tma_load_2d(a, map_a, full, ct * kTileK, p0);
        }
        if (kBmn) {
#pragma unroll
          for (int jb = 0; jb < RP / 64; ++jb) tma_load_2d(b + jb * 8192, map_b, full, jb * 64, ct * kTileK);
        } else {
          tma_load_2d(b, map_b, full, ct * kTileK, 0);
        }
      }
      for (int q = i - 1; q >= 0 && q >= i - kSkStages; --q)
        mbar_wait(bar0 + 8u * (q % kSkStages), (q / kSkStages) & 1, ab, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kTileP, RP, kAmn ? 1 : 0, kBmn ? 1 : 0);
      for (int i = 0; i < nct; ++i) {
        const int slot = i % kSkStages;
        const uint32_t ph = (i / kSkStages) & 1;
        if (!mbar_wait(bar0 + 8u * slot, ph, ab)) break;
        tc_fence_after_sync();
        const uint32_t a = base + slot * S::kStageBytes;
        const uint32_t b = a + S::kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = kAmn ? sw128_desc(a + kk * 2048, 8192, 1024) : sw128_desc(a + kk * 32, 16, 1024);
          const uint64_t bd = kBmn ? sw128_desc(b + kk * 2048, 8192, 1024) : sw128_desc(b + kk * 32, 16, 1024);
          umma_bf16(tmem_d, ad, bd, idesc, (i | kk) != 0 ? 1u : 0u);
        }
        umma_commit(bar0 + 8u * (kSkStages + slot));
      }
      umma_commit(accum_bar);
    }
    __syncwarp();
  } else {
    // epilogue: TMEM lane = tile row; the partial tile goes to shared memory
    bool ok = mbar_wait(accum_bar, 0, ab, false);
    tc_fence_after_sync();
    ok = __all_sync(0xffffffffu, ok && (s_abort == 0));
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    if (ok) {
      const uint32_t dst = base + static_cast<uint32_t>(row * S::kRedStride) * 4u;
#pragma unroll
      for (int c0 = 0; c0 < RP; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem_d + (static_cast<uint32_t>(quarter * 32) << 16) + c0, v);
        tmem_ld_wait();
        const bool live = nct > 0;
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          st_shared_f4(dst + (c0 + j) * 4u, live ? __uint_as_float(v[j]) : 0.f,
                       live ? __uint_as_float(v[j + 1]) : 0.f, live ? __uint_as_float(v[j + 2]) : 0.f,
                       live ? __uint_as_float(v[j + 3]) : 0.f);
      }
    }
  }

  // all partial tiles of the cluster are in shared memory after this barrier
  cluster_sync_all();

  if (warp >= 2 && s_abort == 0) {
    const int t = threadIdx.x - 64;   // 0..127
    const uint32_t rank = cluster_ctarank();
    const int rows_per = kTileP / static_cast<int>(nsplit);
    const int row_begin = static_cast<int>(rank) * rows_per;
    constexpr int kGroups = RP / 4;
    const bool transposed = (MODE == kRed && job == 1);
    for (int e = t; e < rows_per * kGroups; e += 128) {
      int lr, cg;
      if (transposed) {   // dB [r, rows]: consecutive threads take consecutive rows
        cg = e / rows_per;
        lr = e % rows_per;
      } else {
        lr = e / kGroups;
        cg = e % kGroups;
      }
      const int row = row_begin + lr;
      const int grow = p0 + row;
      if (grow >= j_rows) continue;
      const int col = cg * 4;
      const uint32_t local = base + static_cast<uint32_t>(row * S::kRedStride + col) * 4u;
      float4 part[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < static_cast<int>(nsplit)) part[q] = ld_dsmem_v4(map_to_cta(local, q));
      float4 sum = part[0];
#pragma unroll
      for (int q = 1; q < 8; ++q)
        if (q < static_cast<int>(nsplit)) {
          sum.x += part[q].x;
          sum.y += part[q].y;
          sum.z += part[q].z;
          sum.w += part[q].w;
        }
      const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
      if (MODE == kRowsT) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (col + c < p.r) j_out_f32[static_cast<int64_t>(grow) * p.r + col + c] = vals[c];
        *reinterpret_cast<uint2*>(j_out_bf16 + static_cast<int64_t>(grow) * RP + col) = bf16x4_scaled(p.s, sum);
      } else if (MODE == kRowsG) {
        *reinterpret_cast<uint2*>(j_out_bf16 + static_cast<int64_t>(grow) * RP + col) = bf16x4_scaled(p.s, sum);
      } else if (!transposed) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (col + c < p.r) j_out_f32[static_cast<int64_t>(grow) * p.r + col + c] = vals[c];
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (col + c < p.r) j_out_f32[static_cast<int64_t>(col + c) * j_rows + grow] = vals[c];
      }
    }
    if (MODE == kRowsG) {
      // bf16(s*T) for the same rows, from the fp32 T saved by the forward
      for (int e = t; e < rows_per * kGroups; e += 128) {
        const int grow = p0 + row_begin + e / kGroups;
        if (grow >= j_rows) continue;
        const int col = (e % kGroups) * 4;
        float v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          v[c] = (col + c < p.r) ? p.xa[static_cast<int64_t>(grow) * p.r + col + c] : 0.0f;
        *reinterpret_cast<uint2*>(p.s_t + static_cast<int64_t>(grow) * RP + col) =
            bf16x4_scaled(p.s, make_float4(v[0], v[1], v[2], v[3]));
      }
    }
  }

  // nobody leaves while a peer may still read its shared memory
  cluster_sync_all();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_d, RP);
  }
}

// ============================================================== main fused GEMM

constexpr int kMainStages = 4;
constexpr int kMainThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 dequant + epilogue

template <int BN>
struct MainSmem {
  static constexpr int kActBytes = BN * 128;      // BN tokens x 64 contraction
  static constexpr int kWBytes = kTileP * 128;    // 128 features x 64 contraction
  static constexpr int kStageBytes = kActBytes + kWBytes;
  static constexpr int kBarOffset = kMainStages * kStageBytes;
  static constexpr int kBytes = kBarOffset + 256 + 1024;
  static_assert(BN * kTileP * 2 <= kBarOffset, "epilogue staging must fit");
};

struct MainParams {
  const uint8_t* packed;   // NF4 codes of W [N, K]
  const float* absmax;     // [N * K / 64]
  int K;                   // d_in
  int N;                   // d_out
  int num_kt;              // NF4 stages
  int num_lt;              // LoRA stages
  int* status;
};

template <int BN, bool kTrans>
__global__ void __launch_bounds__(kMainThreads, 1)
    lora_main_kernel(const __grid_constant__ CUtensorMap map_act,    // X or dY, box {64, BN}
                     const __grid_constant__ CUtensorMap map_lact,   // bf16(s*T) or bf16(s*G), box {64, BN}
                     const __grid_constant__ CUtensorMap map_lw,     // Y: B [r, N], box {64, 64}; dX: A [K, r], box {64, 128}
                     const __grid_constant__ CUtensorMap map_out,    // Y or dX, box {128, BN}
                     const MainParams p) {
  using S = MainSmem<BN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t bar0 = base + S::kBarOffset;
  // barriers: full_act[st], full_w[st], empty[st], accum
  const uint32_t accum_bar = bar0 + 8u * (3 * kMainStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p0 = blockIdx.x * kTileP;
  const int t0 = blockIdx.y * BN;
  const int total = p.num_kt + p.num_lt;
  Abort ab{&s_abort, p.status};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kMainStages; ++i) {
      mbar_init(bar0 + 8u * i, 1);                          // full_act: TMA bytes
      mbar_init(bar0 + 8u * (kMainStages + i), 4);          // full_w: the 4 warps of one dequant group
      mbar_init(bar0 + 8u * (2 * kMainStages + i), 1);      // empty: MMA commit
    }
    mbar_init(accum_bar, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_act);
    tma_prefetch_map(&map_lact);
    tma_prefetch_map(&map_lw);
    tma_prefetch_map(&map_out);
  }
  if (warp == 1) tmem_alloc(smem_u32(&s_tmem), BN);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_d = s_tmem;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int s = 0;
      for (; s < total; ++s) {
        const int slot = s % kMainStages;
        const uint32_t ph = (s / kMainStages) & 1;
        if (!mbar_wait(bar0 + 8u * (2 * kMainStages + slot), ph ^ 1, ab)) break;
        const uint32_t act = base + slot * S::kStageBytes;
        const uint32_t full = bar0 + 8u * slot;
        if (s < p.num_kt) {
          mbar_arrive_expect_tx(full, S::kActBytes);
          tma_load_2d(act, &map_act, full, s * kTileK, t0);
        } else {
          const int j = s - p.num_kt;
          mbar_arrive_expect_tx(full, S::kActBytes + S::kWBytes);
          tma_load_2d(act, &map_lact, full, j * kTileK, t0);
          if (kTrans) {
            // A [K, r] rows p0..p0+127, LoRA columns 64j..: K-major
            tma_load_2d(act + S::kActBytes, &map_lw, full, j * kTileK, p0);
          } else {
            // B [r, N] rows 64j.. (the LoRA contraction), columns p0..p0+127: MN-major
            tma_load_2d(act + S::kActBytes, &map_lw, full, p0, j * kTileK);
            tma_load_2d(act + S::kActBytes + 8192, &map_lw, full, p0 + 64, j * kTileK);
          }
        }
      }
      for (int q = s - 1; q >= 0 && q >= s - kMainStages; --q)
        mbar_wait(bar0 + 8u * (q % kMainStages), (q / kMainStages) & 1, ab, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      // A operand majorness: Y -- W tile K-major, B tile MN-major; dX -- W tile MN-major, A tile K-major
      constexpr uint32_t idesc_w = umma_idesc_bf16(kTileP, BN, kTrans ? 1 : 0, 0);
      constexpr uint32_t idesc_l = umma_idesc_bf16(kTileP, BN, kTrans ? 0 : 1, 0);
      for (int s = 0; s < total; ++s) {
        const int slot = s % kMainStages;
        const uint32_t ph = (s / kMainStages) & 1;
        if (!mbar_wait(bar0 + 8u * slot, ph, ab)) break;
        if (!mbar_wait(bar0 + 8u * (kMainStages + slot), ph, ab)) break;
        tc_fence_after_sync();
        const uint32_t act = base + slot * S::kStageBytes;
        const uint32_t wt = act + S::kActBytes;
        const bool lora = s >= p.num_kt;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const bool a_mn = (kTrans != lora);
          const uint64_t ad = a_mn ? sw128_desc(wt + kk * 2048, 8192, 1024) : sw128_desc(wt + kk * 32, 16, 1024);
          const uint64_t bd = sw128_desc(act + kk * 32, 16, 1024);
          umma_bf16(tmem_d, ad, bd, lora ? idesc_l : idesc_w, (s | kk) != 0 ? 1u : 0u);
        }
        umma_commit(bar0 + 8u * (2 * kMainStages + slot));
      }
      umma_commit(accum_bar);
    }
    __syncwarp();
  } else {
    // ---------------- NF4 dequantisation into the UMMA A operand
    const int dw = warp - 2;                  // 0..7
    const int grp = dw >> 2;                  // group g converts stages s with s % 2 == g
    const int i = (dw & 3) * 32 + lane;       // operand row written by this thread
    const uint32_t row_off = static_cast<uint32_t>(i) * 128u;
    const uint32_t swz = static_cast<uint32_t>(i & 7);
    const int kblocks = p.K >> 6;
    // absmax index of the 64-element block this thread expands at NF4 stage s
    // (or -1 outside W): Y uses W rows p0.. along K; dX uses W rows 64s.. and
    // the two 64-column blocks of this CTA's 128 features.
    auto block_of = [&](int s) -> int64_t {
      int n, kb;
      if (!kTrans) {
        n = p0 + i;
        kb = s;
      } else {
        n = s * 64 + (i & 63);
        kb = (p0 >> 6) + (i >> 6);
      }
      if (n >= p.N || kb >= kblocks) return -1;
      return static_cast<int64_t>(n) * kblocks + kb;
    };
    const uint8_t* packed = p.packed;
    const float* absmax = p.absmax;

    // codes and absmax of this thread's block, loaded two of its iterations ahead
    struct Pending {
      uint4 lo, hi;
      float am;
      bool valid;
    };
    auto fetch = [&](int s) -> Pending {
      Pending f;
      f.lo = make_uint4(0u, 0u, 0u, 0u);
      f.hi = f.lo;
      f.am = 0.0f;
      f.valid = false;
      if (s < p.num_kt) {
        const int64_t b = block_of(s);
        if (b >= 0) {
          f.lo = ldg_nc_v4(packed + 32 * b);
          f.hi = ldg_nc_v4(packed + 32 * b + 16);
          f.am = ldg_nc_f32(absmax + b);
          f.valid = true;
        }
      }
      return f;
    };
    Pending cur = fetch(grp);
    Pending nxt = fetch(grp + 2);
    for (int s = grp; s < total; s += 2) {
      const Pending later = fetch(s + 4);
      const int slot = s % kMainStages;
      const uint32_t ph = (s / kMainStages) & 1;
      // one lane waits for the slot to be free, the warp follows (warp-uniform exit on abort)
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bar0 + 8u * (2 * kMainStages + slot), ph ^ 1, ab);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (s < p.num_kt) {
        const uint32_t dst = base + slot * S::kStageBytes + S::kActBytes + row_off;
        if (cur.valid) {
          const Nf4BlockTable tab = nf4_block_table(cur.am);
          const uint32_t words[8] = {cur.lo.x, cur.lo.y, cur.lo.z, cur.lo.w,
                                     cur.hi.x, cur.hi.y, cur.hi.z, cur.hi.w};
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_v4(dst + ((c ^ swz) << 4), nf4_expand8(words[c], tab));
        } else {
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_v4(dst + (c << 4), make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar0 + 8u * (kMainStages + slot));
      cur = nxt;
      nxt = later;
    }

    // ---------------- epilogue: TMEM -> bf16 -> shared staging [BN tokens][128 features] -> TMA store
    bool ok = mbar_wait(accum_bar, 0, ab, false);
    tc_fence_after_sync();
    ok = __all_sync(0xffffffffu, ok && (s_abort == 0));
    const int quarter = warp & 3;
    const int half = dw >> 2;
    const int prow = quarter * 32 + lane;
    if (ok) {
      for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem_d + (static_cast<uint32_t>(quarter * 32) << 16) + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(v[j]));
          st_shared_u16(base + static_cast<uint32_t>(c0 + j) * (kTileP * 2) + prow * 2,
                        *reinterpret_cast<const uint16_t*>(&h));
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (threadIdx.x == 64 && s_abort == 0 && ok) {
      tma_store_2d(&map_out, base, p0, t0);
      tma_store_commit();
      tma_store_wait_all();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_d, BN);
  }
}

// ============================================================== host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 2-D map over a row-major [outer, inner] tensor.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* gaddr, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              bool swizzle128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(m, dt, 2, const_cast<void*>(gaddr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool map_bf16(CUtensorMap* m, const void* g, uint64_t cols, uint64_t rows, uint32_t box_c,
              uint32_t box_r, bool sw) {
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g, cols, rows, cols * 2, box_c, box_r, sw);
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

// Contraction split across a cluster: the largest power of two <= 8 that keeps
// tiles * split within one wave and leaves every CTA at least one tile.
int pick_split(int tiles, int num_ct) {
  const int sms = sm_count();
  int s = 1;
  while (s < 8 && tiles * (2 * s) <= sms && 2 * s <= num_ct) s *= 2;
  return s;
}

template <typename Kern>
cudaError_t set_smem(Kern k, int bytes) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

constexpr int skinny_kind(int mode) {
  return mode == kRowsT ? kKindRowsT : mode == kRowsG ? kKindRowsG : kKindRed;
}

template <int MODE, int RP>
cudaError_t launch_skinny_rp(const CUtensorMap (&maps)[4], const SkinnyParams& sp, int tiles,
                             int split, cudaStream_t stream) {
  auto kern = lora_skinny_kernel<MODE, RP>;
  cudaError_t e = set_smem(kern, SkinnySmem<RP>::kBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, split, 1);
  cfg.blockDim = dim3(kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = SkinnySmem<RP>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = split;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchScope scope(skinny_kind(MODE), stream);
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], sp);
}

template <int MODE>
cudaError_t launch_skinny(int rp, const CUtensorMap (&maps)[4], const SkinnyParams& sp, int tiles,
                          int split, cudaStream_t stream) {
  if (rp == 64) return launch_skinny_rp<MODE, 64>(maps, sp, tiles, split, stream);
  return launch_skinny_rp<MODE, 128>(maps, sp, tiles, split, stream);
}

template <int BN, bool kTrans>
cudaError_t launch_main_bn(const CUtensorMap& ma, const CUtensorMap& ml, const CUtensorMap& mw,
                           const CUtensorMap& mo, const MainParams& mp, int P, int M,
                           cudaStream_t stream) {
  auto kern = lora_main_kernel<BN, kTrans>;
  cudaError_t e = set_smem(kern, MainSmem<BN>::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((P + kTileP - 1) / kTileP, (M + BN - 1) / BN, 1);
  LaunchScope scope(kTrans ? kKindMainDx : kKindMainFwd, stream);
  kern<<<grid, kMainThreads, MainSmem<BN>::kBytes, stream>>>(ma, ml, mw, mo, mp);
  return cudaGetLastError();
}

int pick_bn(int M) { return M <= 64 ? 64 : (M <= 128 ? 128 : 256); }

// The low-rank weight the kernels read: A itself when its rows are 16-byte
// multiples (r % 8 == 0), else the zero-padded copy [K, rp] in the workspace.
struct LowRankA {
  const uint16_t* ptr;
  int cols;
};

LowRankA low_rank_a(const LayerDims& d, const uint16_t* A, const Workspace& ws) {
  if (d.r % 8 == 0) return {A, d.r};
  return {ws.a_pad, d.rp};
}

// One fused GEMM: out [M, P] = act [M, C] . W_side^T + lact [M, rp] . (low-rank side)^T.
//   Y : act = X,  W_side = W_deq,      lact = bf16(s*T), low-rank side = B^T (read from B [r, N])
//   dX: act = dY, W_side = W_deq^T,    lact = bf16(s*G), low-rank side = A   (read from A [K, r])
template <bool kTrans>
cudaError_t launch_main(const LayerDims& d, const uint16_t* act, const uint16_t* lact,
                        const uint16_t* lw, int lw_cols, uint16_t* out, const uint8_t* packed,
                        const float* absmax, int* status, cudaStream_t stream) {
  const int P = kTrans ? d.K : d.N;     // output features
  const int C = kTrans ? d.N : d.K;     // contraction length of the NF4 part
  const int bn = pick_bn(d.M);
  CUtensorMap ma, ml, mw, mo;
  bool ok = map_bf16(&ma, act, C, d.M, 64, bn, true) && map_bf16(&ml, lact, d.rp, d.M, 64, bn, true) &&
            map_bf16(&mo, out, P, d.M, kTileP, bn, false);
  if (kTrans) ok = ok && map_bf16(&mw, lw, lw_cols, d.K, 64, kTileP, true);   // A [K, r]
  else ok = ok && map_bf16(&mw, lw, d.N, d.r, 64, 64, true);                   // B [r, N]
  if (!ok) return cudaErrorInvalidValue;
  MainParams mp;
  mp.packed = packed;
  mp.absmax = absmax;
  mp.K = d.K;
  mp.N = d.N;
  mp.num_kt = (C + kTileK - 1) / kTileK;
  mp.num_lt = d.rp / kTileK;
  mp.status = status;
  if (bn == 64) return launch_main_bn<64, kTrans>(ma, ml, mw, mo, mp, P, d.M, stream);
  if (bn == 128) return launch_main_bn<128, kTrans>(ma, ml, mw, mo, mp, P, d.M, stream);
  return launch_main_bn<256, kTrans>(ma, ml, mw, mo, mp, P, d.M, stream);
}

// Pads A to [K, rp] (only needed when r % 8 != 0).
cudaError_t launch_pad_a(const LayerDims& d, const uint16_t* A, const Workspace& ws,
                         cudaStream_t stream) {
  if (d.r % 8 == 0) return cudaSuccess;
  PrepParams pp = {};
  pp.A = A;
  pp.a_pad = ws.a_pad;
  pp.n_apad = static_cast<int64_t>(d.K) * d.rp;
  pp.N = d.N;
  pp.r = d.r;
  pp.rp = d.rp;
  pp.s = d.s;
  const int64_t want = (pp.n_apad + 255) / 256;
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sm_count()) * 8));
  LaunchScope scope(kKindPrep, stream);
  lora_prep_kernel<<<grid, 256, 0, stream>>>(pp);
  return cudaGetLastError();
}

size_t align_up(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

}  // namespace

size_t workspace_bytes(const LayerDims& d) {
  const size_t rp = static_cast<size_t>(d.rp);
  return align_up(static_cast<size_t>(d.K) * rp * 2) + 2 * align_up(static_cast<size_t>(d.M) * rp * 2);
}

Workspace carve_workspace(const LayerDims& d, void* base) {
  const size_t rp = static_cast<size_t>(d.rp);
  uint8_t* b = static_cast<uint8_t*>(base);
  Workspace w;
  w.a_pad = reinterpret_cast<uint16_t*>(b);
  b += align_up(static_cast<size_t>(d.K) * rp * 2);
  w.s_t = reinterpret_cast<uint16_t*>(b);
  b += align_up(static_cast<size_t>(d.M) * rp * 2);
  w.s_g = reinterpret_cast<uint16_t*>(b);
  return w;
}

cudaError_t run_forward(const LayerDims& d, const uint16_t* X, const uint8_t* packed,
                        const float* absmax, const uint16_t* A, const uint16_t* B, uint16_t* Y,
                        float* XA, const Workspace& ws, int* status, cudaStream_t stream) {
  cudaError_t e = launch_pad_a(d, A, ws, stream);
  if (e != cudaSuccess) return e;
  const LowRankA la = low_rank_a(d, A, ws);
  // T = X . A  (fp32, saved) and bf16(s*T)
  {
    CUtensorMap maps[4];
    if (!map_bf16(&maps[0], X, d.K, d.M, 64, kTileP, true) ||
        !map_bf16(&maps[1], la.ptr, la.cols, d.K, 64, 64, true))
      return cudaErrorInvalidValue;
    maps[2] = maps[0];
    maps[3] = maps[1];
    SkinnyParams sp = {};
    sp.r = d.r;
    sp.num_ct = d.K / kTileK;
    sp.s = d.s;
    sp.job[0].rows = d.M;
    sp.job[0].tiles = (d.M + kTileP - 1) / kTileP;
    sp.job[0].out_f32 = XA;
    sp.job[0].out_bf16 = ws.s_t;
    sp.status = status;
    const int tiles = sp.job[0].tiles;
    e = launch_skinny<kRowsT>(d.rp, maps, sp, tiles, pick_split(tiles, sp.num_ct), stream);
    if (e != cudaSuccess) return e;
  }
  return launch_main<false>(d, X, ws.s_t, B, d.r, Y, packed, absmax, status, stream);
}

cudaError_t run_backward(const LayerDims& d, const uint16_t* X, const uint16_t* dY,
                         const uint8_t* packed, const float* absmax, const uint16_t* A,
                         const uint16_t* B, const float* XA, uint16_t* dX, float* dA, float* dB,
                         const Workspace& ws, int* status, cudaStream_t stream) {
  cudaError_t e = launch_pad_a(d, A, ws, stream);
  if (e != cudaSuccess) return e;
  const LowRankA la = low_rank_a(d, A, ws);
  // bf16(s * dY . B^T), and bf16(s*T) from the saved T
  {
    CUtensorMap maps[4];
    if (!map_bf16(&maps[0], dY, d.N, d.M, 64, kTileP, true) ||
        !map_bf16(&maps[1], B, d.N, d.r, 64, d.rp, true))
      return cudaErrorInvalidValue;
    maps[2] = maps[0];
    maps[3] = maps[1];
    SkinnyParams sp = {};
    sp.r = d.r;
    sp.num_ct = (d.N + kTileK - 1) / kTileK;
    sp.s = d.s;
    sp.job[0].rows = d.M;
    sp.job[0].tiles = (d.M + kTileP - 1) / kTileP;
    sp.job[0].out_bf16 = ws.s_g;
    sp.xa = XA;
    sp.s_t = ws.s_t;
    sp.status = status;
    const int tiles = sp.job[0].tiles;
    e = launch_skinny<kRowsG>(d.rp, maps, sp, tiles, pick_split(tiles, sp.num_ct), stream);
    if (e != cudaSuccess) return e;
  }
  // dA = X^T . bf16(s*G)  -> [K, r]   and   dB = bf16(s*T)^T . dY  -> [r, N], one launch
  {
    CUtensorMap maps[4];
    if (!map_bf16(&maps[0], X, d.K, d.M, 64, 64, true) || !map_bf16(&maps[1], ws.s_g, d.rp, d.M, 64, 64, true) ||
        !map_bf16(&maps[2], dY, d.N, d.M, 64, 64, true) || !map_bf16(&maps[3], ws.s_t, d.rp, d.M, 64, 64, true))
      return cudaErrorInvalidValue;
    SkinnyParams sp = {};
    sp.r = d.r;
    sp.num_ct = (d.M + kTileK - 1) / kTileK;
    sp.job[0].rows = d.K;
    sp.job[0].tiles = (d.K + kTileP - 1) / kTileP;
    sp.job[0].out_f32 = dA;
    sp.job[1].rows = d.N;
    sp.job[1].tiles = (d.N + kTileP - 1) / kTileP;
    sp.job[1].out_f32 = dB;
    sp.status = status;
    const int tiles = sp.job[0].tiles + sp.job[1].tiles;
    e = launch_skinny<kRed>(d.rp, maps, sp, tiles, pick_split(tiles, sp.num_ct), stream);
    if (e != cudaSuccess) return e;
  }
  if (dX == nullptr) return cudaSuccess;
  return launch_main<true>(d, dY, ws.s_g, la.ptr, la.cols, dX, packed, absmax, status, stream);
}

}  // namespace qlora
