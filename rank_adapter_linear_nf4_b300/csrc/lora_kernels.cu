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

constexpr int kSkThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue

template <int RP>
struct SkinnySmem {
  static constexpr int kStages = RP == 64 ? 8 : RP == 128 ? 6 : 4;   // as many as fit: keeps HBM reads in flight
  static constexpr int kABytes = kTileP * 128;   // 128 rows x 64 bf16
  static constexpr int kBBytes = RP * 128;       // RP columns x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = kStages * kStageBytes;
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
  int* zero;           // rows modes: split-tile counters of the main kernel that follows
  int n_zero;
  int grp_n;           // kRed job 1 (dB) of stacked projections: only the diagonal blocks,
  int grp_width;       // grp_width rank rows of group g for the features of g
  int grp_end[kMaxLoraGroups];
  int wait_first;      // launched with programmatic serialisation as a call's first kernel:
                       // wait for the previous kernel before touching global memory
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

template <int MODE, int RP, int NSPLIT>
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
  const uint32_t accum_bar = bar0 + 8u * (2 * S::kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int job = (MODE == kRed && static_cast<int>(blockIdx.x) >= p.job[0].tiles) ? 1 : 0;
  // job fields picked with selects (a dynamic index into the parameter struct would spill it)
  const int j_rows = job ? p.job[1].rows : p.job[0].rows;
  float* const j_out_f32 = job ? p.job[1].out_f32 : p.job[0].out_f32;
  uint16_t* const j_out_bf16 = p.job[0].out_bf16;
  const CUtensorMap* map_a = job ? &map_a1 : &map_a0;
  const CUtensorMap* map_b = job ? &map_b1 : &map_b0;
  const int p0 = (static_cast<int>(blockIdx.x) - (job ? p.job[0].tiles : 0)) * kTileP;
  constexpr uint32_t nsplit = NSPLIT;   // == gridDim.y == cluster size
  const uint32_t split = blockIdx.y;
  const int ct_begin = static_cast<int>((static_cast<int64_t>(p.num_ct) * split) / nsplit);
  const int ct_end = static_cast<int>((static_cast<int64_t>(p.num_ct) * (split + 1)) / nsplit);
  const int nct = ct_end - ct_begin;
  Abort ab{&s_abort, p.status};
  // the low-rank columns this tile contracts against: all of them, or (dB of
  // stacked projections) the group that owns the tile's features
  int lr_off = 0, lr_n = RP, lr_valid = p.r;
  if (MODE == kRed && job == 1 && p.grp_n > 0) {
    int g = 0;
    while (g + 1 < p.grp_n && p0 >= p.grp_end[g]) ++g;
    lr_off = g * p.grp_width;
    lr_n = p.grp_width;
    lr_valid = p.grp_width;
  }

  if (threadIdx.x == 0) {
    // a dependent kernel may be scheduled now: it waits (griddepcontrol.wait)
    // before it reads anything this kernel writes.  It does read the call's
    // inputs before that wait, so a kernel that itself started early lets it
    // go only after its own wait (below).
    if (!p.wait_first) griddep_launch_dependents();
    s_abort = 0;
    for (int i = 0; i < S::kStages; ++i) {
      mbar_init(bar0 + 8u * i, 1);                    // full
      mbar_init(bar0 + 8u * (S::kStages + i), 1);      // empty
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
  // as a call's first kernel this one may start while the previous kernel on the
  // stream runs: the set-up above overlaps it, the reads and writes below wait
  if (p.wait_first) {
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();
  }
  if (MODE != kRed && blockIdx.x == 0 && blockIdx.y == 0) {
    // the main kernel after this one counts finished pieces of its split tiles
    // from zero; it reads the counters only after waiting for this kernel
    for (int i = static_cast<int>(threadIdx.x); i < p.n_zero; i += kSkThreads) p.zero[i] = 0;
  }

  if (warp == 0) {
    if (lane == 0) {
      int i = 0;
      for (; i < nct; ++i) {
        const int slot = i % S::kStages;
        const uint32_t ph = (i / S::kStages) & 1;
        if (!mbar_wait(bar0 + 8u * (S::kStages + slot), ph ^ 1, ab)) break;
        const int ct = ct_begin + i;
        const uint32_t a = base + slot * S::kStageBytes;
        const uint32_t b = a + S::kABytes;
        const uint32_t full = bar0 + 8u * slot;
        mbar_arrive_expect_tx(full, kBmn ? S::kABytes + (lr_n / 64) * 8192 : S::kStageBytes);
        if (kAmn) {
          tma_load_2d(a, map_a, full, p0, ct * kTileK);
          tma_load_2d(a + 8192, map_a, full, p0 + 64, ct * kTileK);
        } else {
          tma_load_2d(a, map_a, full, ct * kTileK, p0);
        }
        if (kBmn) {
#pragma unroll
          for (int jb = 0; jb < RP / 64; ++jb)
            if (jb * 64 < lr_n) tma_load_2d(b + jb * 8192, map_b, full, lr_off + jb * 64, ct * kTileK);
        } else {
          tma_load_2d(b, map_b, full, ct * kTileK, 0);
        }
      }
      for (int q = i - 1; q >= 0 && q >= i - S::kStages; --q)
        mbar_wait(bar0 + 8u * (q % S::kStages), (q / S::kStages) & 1, ab, false);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kTileP, lr_n, kAmn ? 1 : 0, kBmn ? 1 : 0);
      for (int i = 0; i < nct; ++i) {
        const int slot = i % S::kStages;
        const uint32_t ph = (i / S::kStages) & 1;
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
        umma_commit(bar0 + 8u * (S::kStages + slot));
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
    // Sum the NSPLIT partial tiles in rank order.  Every remote load of a pass is
    // issued before any is consumed, so the pass costs one DSMEM round trip.
    const int t = threadIdx.x - 64;   // 0..127
    const uint32_t rank = cluster_ctarank();
    constexpr int kRowsPer = kTileP / NSPLIT;
    constexpr int kGroups = RP / 4;                      // float4 column groups per row
    constexpr int kItemsPerPass = 16 / NSPLIT;           // (row, group) items per thread per pass
    constexpr int kPasses = (kRowsPer * kGroups) / (128 * kItemsPerPass);
    const int row_begin = static_cast<int>(rank) * kRowsPer;
    const bool transposed = (MODE == kRed && job == 1);
#pragma unroll
    for (int pass = 0; pass < kPasses; ++pass) {
      float4 part[kItemsPerPass][NSPLIT];
      int rows[kItemsPerPass], cols[kItemsPerPass];
#pragma unroll
      for (int it = 0; it < kItemsPerPass; ++it) {
        const int e = t + (pass * kItemsPerPass + it) * 128;
        int lr, cg;
        if (transposed) {   // dB [r, rows]: consecutive threads take consecutive rows
          cg = e / kRowsPer;
          lr = e % kRowsPer;
        } else {
          lr = e / kGroups;
          cg = e % kGroups;
        }
        rows[it] = row_begin + lr;
        cols[it] = cg * 4;
        const uint32_t local = base + static_cast<uint32_t>(rows[it] * S::kRedStride + cols[it]) * 4u;
#pragma unroll
        for (int q = 0; q < NSPLIT; ++q) part[it][q] = ld_dsmem_v4(map_to_cta(local, q));
      }
#pragma unroll
      for (int it = 0; it < kItemsPerPass; ++it) {
        const int grow = p0 + rows[it];
        if (grow >= j_rows) continue;
        const int col = cols[it];
        float4 sum = part[it][0];
#pragma unroll
        for (int q = 1; q < NSPLIT; ++q) {
          sum.x += part[it][q].x;
          sum.y += part[it][q].y;
          sum.z += part[it][q].z;
          sum.w += part[it][q].w;
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
            if (col + c < lr_valid) j_out_f32[static_cast<int64_t>(lr_off + col + c) * j_rows + grow] = vals[c];
        }
      }
    }
    if (MODE == kRowsG) {
      // bf16(s*T) for the same rows, from the fp32 T saved by the forward (loads first, then stores)
#pragma unroll
      for (int pass = 0; pass < kPasses; ++pass) {
        float v[kItemsPerPass][4];
#pragma unroll
        for (int it = 0; it < kItemsPerPass; ++it) {
          const int e = t + (pass * kItemsPerPass + it) * 128;
          const int grow = p0 + row_begin + e / kGroups;
          const int col = (e % kGroups) * 4;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            v[it][c] = (grow < j_rows && col + c < p.r) ? __ldg(p.xa + static_cast<int64_t>(grow) * p.r + col + c) : 0.0f;
        }
#pragma unroll
        for (int it = 0; it < kItemsPerPass; ++it) {
          const int e = t + (pass * kItemsPerPass + it) * 128;
          const int grow = p0 + row_begin + e / kGroups;
          if (grow >= j_rows) continue;
          const int col = (e % kGroups) * 4;
          *reinterpret_cast<uint2*>(p.s_t + static_cast<int64_t>(grow) * RP + col) =
              bf16x4_scaled(p.s, make_float4(v[it][0], v[it][1], v[it][2], v[it][3]));
        }
      }
    }
  }

  // nobody leaves while a peer may still read its shared memory
  cluster_sync_all();
  // when launched with programmatic serialisation this kernel may overlap the one
  // before it; finishing only after that one has finished keeps the stream order
  // seen by later work (a later normal launch waits for this kernel alone)
  griddep_wait();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_d, RP);
  }
}

// ============================================================== main fused GEMM

constexpr int kEpiChunk = 32;        // tokens per epilogue store
constexpr int kMinSkStages = 16;     // fewest stages a CTA takes in the split remainder
// warp 0: TMA for the token operand; warp 1: MMA (in the odd CTA of a pair: the relay of its
// stages to the even CTA, whose thread issues the pair's MMAs); warps 2-9: dequant; warps 10-13:
// epilogue; warp 14: TMA for the NF4 codes and absmax (its own ring, so code latency never holds
// up operand loads)
constexpr int kMainThreads = 480;

// Ring depths, as deep as shared memory allows.  With few tokens per tile the
// kernel streams the weight, and each stage is short: the operand ring must
// cover a TMA load plus an MMA round trip, the code ring the HBM latency.
constexpr int main_stages(int bn) { return bn <= 64 ? 8 : 4; }
constexpr int raw_stages(int bn) { return (bn == 32 || bn == 128) ? 8 : 4; }

// kPair: the CTA pair's UMMA (cta_group::2, M = 256) covers 256 output
// features (128 per CTA, each CTA expanding its own W rows) and the BN tokens
// of the tile, each CTA staging half of them.  Per SM a stage is then 32 KB
// instead of 48 (a ring of six fits instead of four), and the tensor core
// reads and TMA writes half the token rows: fewer shared-memory bytes per
// flop, which also lowers the power drawn per flop.
template <int BN, bool kPair = false>
struct MainSmem {
  static constexpr int kActRows = kPair ? BN / 2 : BN;   // token rows staged by this CTA
  // a pair's 32 KB stages leave room for six in the ring (slots are g % kStages)
  static constexpr int kStages = kPair ? 6 : main_stages(kActRows);
  static constexpr int kRaw = kPair ? 4 : raw_stages(kActRows);
  // one UMMA of N = BN per K step (at most 256); two TMEM accumulators of BN
  // columns, so the epilogue of one piece overlaps the main loop of the next
  static constexpr int kMmaN = BN < 256 ? BN : 256;
  static constexpr int kHalves = kPair ? 1 : BN / kMmaN;
  static constexpr int kAccs = 2;
  static constexpr int kActBytes = kActRows * 128;   // staged tokens x 64 contraction
  static constexpr int kWBytes = kTileP * 128;    // 128 features x 64 contraction
  static constexpr int kStageBytes = kActBytes + kWBytes;
  static constexpr int kCodeBytes = 4096;         // Y: 128 rows x 32 B; dX: 64 rows x 64 B
  static constexpr int kAbsBytes = 2048;          // Y: 128 rows x 4 fp32; dX: 64 rows x 4 fp32
  static constexpr int kRawBytes = kCodeBytes + kAbsBytes;
  static constexpr int kRawOffset = kStages * kStageBytes;
  static constexpr int kChunkBytes = kEpiChunk * kTileP * 2;   // two [32 tokens][64 features] halves
  static constexpr int kStagingOffset = kRawOffset + kRaw * kRawBytes;
  static constexpr int kBarOffset = kStagingOffset + kChunkBytes;
  static constexpr int kBarBytes = 8 * (3 * kStages + 2 * kRaw + 5);
  static constexpr int kBytes = kBarOffset + 512 + 1024;
  static_assert(kBarBytes <= 512, "barrier area");
  static_assert(kBytes <= 232448, "shared memory budget");
};

// Work schedule of the persistent grid.  Tiles (128 features x BN tokens,
// tile id = token_tile * p_tiles + feature_tile) are cut into stages: the NF4
// stages of the contraction, then the LoRA stages.
//   * whole tiles: CTA c takes tiles c, c + grid, ... below dp_tiles;
//   * split remainder: the stages of tiles dp_tiles.. are laid end to end and
//     cut into sk_ctas equal ranges, one per CTA 0..sk_ctas-1.  A range covers
//     pieces of one or more tiles; a piece that is not a whole tile writes an
//     fp32 partial tile, and the last piece of a tile to finish (a per-tile
//     counter) adds the partials in contraction order and stores the tile.
struct MainParams {
  const float* absmax;     // [N * K / 64], read directly when kAbsTma is false
  float* partials;         // [2 * sk_ctas][BN][128] fp32 partial tiles (split remainder only)
  int* counters;           // [sk_tiles] pieces finished per split tile; zero at launch
  int M;                   // tokens
  int K;                   // d_in
  int N;                   // d_out
  int num_kt;              // NF4 stages per tile
  int num_lt;              // LoRA stages per tile
  int p_tiles;             // output-feature tiles of 128
  int t_tiles;             // token tiles of BN
  int dp_tiles;            // tiles taken whole, round robin
  int dp_rounds;           // ceil(dp_tiles / grid)
  int sk_tiles;            // tiles dp_tiles .. dp_tiles + sk_tiles - 1 are split
  int sk_ctas;             // CTAs sharing the split remainder
  int debug_stall;         // test hook: the token producer issues nothing, so every wait runs out
  // Y of stacked projections with separate low-rank blocks: the tile at output
  // feature p0 runs the LoRA stages of its group, starting at stage grp_lt0 * g
  int grp_n;
  int grp_lt0;
  int grp_end[kMaxLoraGroups];
  // SwiGLU gate fused into the epilogue (rows of W and columns of the output
  // interleaved in 64-row chunks: [gate 0..63 | up 0..63 | gate 64..127 | ...]):
  //   Y (gate_fwd):  besides gu = the layer's output, h = silu(g) * u via map_h;
  //   dX (gate_bwd): dh = the layer's dX is not stored; dgu, the gate's backward
  //                  in the layout of gu, is written from dh and gu.
  int gate;
  const uint16_t* gu;      // gate_bwd: [M, 2K] bf16 (the forward's gu)
  uint16_t* dgu;           // gate_bwd: [M, 2K] bf16
  int* status;
};

__device__ __forceinline__ float gate_sigmoid(float x) { return 1.f / (1.f + expf(-x)); }

// Piece `idx` of this CTA's work: tile and stage range [sb, se).  Order: the
// first whole-tile round, then the split pieces, then the other whole-tile
// rounds -- the pieces' fixups then overlap the main loop of later tiles, and
// the LoRA stages in the pieces find the previous kernel finished.
__device__ __forceinline__ bool main_piece(const MainParams& p, int cta, int grid, int idx, int& tile,
                                           int& sb, int& se) {
  const int total = p.num_kt + p.num_lt;
  const int dp_first = p.dp_rounds > 0 ? 1 : 0;
  int n_sk = 0;
  int64_t lo = 0, hi = 0;
  if (cta < p.sk_ctas) {
    const int64_t len = static_cast<int64_t>(p.sk_tiles) * total;
    lo = len * cta / p.sk_ctas;
    hi = len * (cta + 1) / p.sk_ctas;
    if (lo < hi) n_sk = static_cast<int>((hi - 1) / total - lo / total) + 1;
  }
  if (idx >= dp_first && idx < dp_first + n_sk) {
    const int j = static_cast<int>(lo / total) + (idx - dp_first);
    tile = p.dp_tiles + j;
    sb = static_cast<int>(max(lo - static_cast<int64_t>(j) * total, int64_t(0)));
    se = static_cast<int>(min(hi - static_cast<int64_t>(j) * total, static_cast<int64_t>(total)));
    return true;
  }
  const int round = idx < dp_first ? 0 : idx - n_sk;
  if (round >= p.dp_rounds) return false;
  tile = cta + round * grid;
  sb = 0;
  se = total;
  // with a split remainder every CTA has exactly dp_rounds whole tiles; without
  // one, the last round may be short
  return tile < p.dp_tiles;
}

// The CTA whose split range holds stage x of the remainder.
__device__ __forceinline__ int sk_owner(const MainParams& p, int64_t x) {
  const int64_t len = static_cast<int64_t>(p.sk_tiles) * (p.num_kt + p.num_lt);
  return static_cast<int>(((x + 1) * p.sk_ctas - 1) / len);
}

// Partial-tile slot of CTA c's piece of split tile j: 0 for the first tile of
// its range, 1 for the last (a range holds at most two pieces that are not
// whole tiles).
// With CTA pairs the split ranges belong to pairs and each CTA of pair c
// (rank 0 or 1) has its own two slots.
template <int BN, bool kPair>
__device__ __forceinline__ float* sk_slot(const MainParams& p, int c, int j, int rank) {
  const int total = p.num_kt + p.num_lt;
  const int64_t len = static_cast<int64_t>(p.sk_tiles) * total;
  const int first = static_cast<int>((len * c / p.sk_ctas) / total);
  const int owner = kPair ? 2 * c + rank : c;
  return p.partials + static_cast<int64_t>(2 * owner + (j == first ? 0 : 1)) * (kTileP * BN);
}

// Walks this CTA's stages one at a time (or n at a time) across its pieces.
struct StageCursor {
  int idx, tile, sb, se, s;
  bool valid;
  __device__ __forceinline__ void init(const MainParams& p, int cta, int grid) {
    idx = 0;
    valid = main_piece(p, cta, grid, 0, tile, sb, se);
    s = sb;
  }
  __device__ __forceinline__ void advance(const MainParams& p, int cta, int grid, int n) {
    s += n;
    while (valid && s >= se) {
      const int carry = s - se;
      ++idx;
      valid = main_piece(p, cta, grid, idx, tile, sb, se);
      s = sb + carry;
    }
  }
};

// Partial tiles go through L2 only (another SM reads them).
__device__ __forceinline__ void st_global_cg_f32(float* ptr, float v) {
  asm volatile("st.global.cg.f32 [%0], %1;" ::"l"(ptr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_global_cg_f32(const float* ptr) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(ptr) : "memory");
  return v;
}

// Persistent, one CTA per SM.  Two TMEM accumulators let the epilogue of one
// piece overlap the main loop of the next.  NF4 codes (and, when kAbsTma, the
// absmax values) of each stage arrive by TMA in a ring of their own; TMA
// zero-fills rows and columns outside W, so outside W the dequantised operand
// is zero without per-thread bounds checks.
template <int BN, bool kTrans, bool kAbsTma, bool kPair>
__global__ void __launch_bounds__(kMainThreads, 1)
    lora_main_kernel(const __grid_constant__ CUtensorMap map_act,    // X or dY, box {64, BN}
                     const __grid_constant__ CUtensorMap map_lact,   // bf16(s*T) or bf16(s*G), box {64, BN}
                     const __grid_constant__ CUtensorMap map_lw,     // Y: B [r, N], box {64, 64}; dX: A [K, r], box {64, 128}
                     const __grid_constant__ CUtensorMap map_out,    // Y or dX, box {64, 32}, 128-B swizzle
                     const __grid_constant__ CUtensorMap map_code,   // packed [N, K/2] bytes; Y box {32, 128}, dX box {64, 64}
                     const __grid_constant__ CUtensorMap map_abs,    // absmax [N, K/64]; Y box {4, 128}, dX box {4, 64}
                     const __grid_constant__ CUtensorMap map_h,      // gate_fwd: h [M, N/2], box {64, 32}, 128-B swizzle
                     const MainParams p) {
  using S = MainSmem<BN, kPair>;
  constexpr int kMainStages = S::kStages;
  constexpr int kRaw = S::kRaw;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_last;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t bar0 = base + S::kBarOffset;
  // full(i): the stage's token tile (TMA bytes, one producer arrival) and its W
  // tile (one arrival per dequant warp of the group) are both in place
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (kMainStages + i); };
  auto raw_full = [&](int i) { return bar0 + 8u * (2 * kMainStages + i); };
  auto raw_empty = [&](int i) { return bar0 + 8u * (2 * kMainStages + kRaw + i); };
  auto tmem_full = [&](int a) { return bar0 + 8u * (2 * kMainStages + 2 * kRaw + a); };
  auto tmem_empty = [&](int a) { return bar0 + 8u * (2 * kMainStages + 2 * kRaw + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kMainStages + 2 * kRaw + 4);
  // pair only, in the even CTA: the odd CTA's stage i is in place too
  auto pfull = [&](int i) { return bar0 + 8u * (2 * kMainStages + 2 * kRaw + 5 + i); };
  auto raw_slot = [&](int i) { return base + S::kRawOffset + static_cast<uint32_t>(i * S::kRawBytes); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = p.num_kt + p.num_lt;
  // schedule units: CTAs, or CTA pairs (cluster of two; rank 0 issues the UMMAs)
  const int rank = kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const int cta = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int grid = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // first output feature of this CTA's rows of a tile
  auto feat0 = [&](int tile) { return (tile % p.p_tiles) * (kPair ? 2 * kTileP : kTileP) + rank * kTileP; };
  int g_end = 0;   // stages this CTA runs
  {
    int tile, sb, se;
    for (int idx = 0; main_piece(p, cta, grid, idx, tile, sb, se); ++idx) g_end += se - sb;
  }
  Abort ab{&s_abort, p.status};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kMainStages; ++i) {
      mbar_init(full(i), 5);        // producer (with TMA bytes) + the 4 warps of one dequant group
      mbar_init(empty(i), 1);       // MMA commit
    }
    for (int i = 0; i < kRaw; ++i) {
      mbar_init(raw_full(i), 1);    // TMA transaction bytes (or a plain arrive for LoRA stages)
      mbar_init(raw_empty(i), 4);   // the 4 warps of the group that reads the slot
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tmem_full(a), 1);                // MMA commit
      mbar_init(tmem_empty(a), kPair ? 8 : 4);   // the epilogue warps (of both CTAs of a pair)
    }
    mbar_init(drain_bar, 1);
    if (kPair)
      for (int i = 0; i < kMainStages; ++i) mbar_init(pfull(i), 1);   // the odd CTA's relay
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_act);
    tma_prefetch_map(&map_lact);
    tma_prefetch_map(&map_lw);
    tma_prefetch_map(&map_out);
    if (!kTrans && p.gate) tma_prefetch_map(&map_h);
    tma_prefetch_map(&map_code);
    if (kAbsTma) tma_prefetch_map(&map_abs);
  }
  if (warp == 1) {
    if (kPair) tmem_alloc_pair(smem_u32(&s_tmem), S::kAccs * BN);
    else tmem_alloc(smem_u32(&s_tmem), S::kAccs * BN);
  }
  tc_fence_before_sync();
  __syncthreads();
  // a pair: the peer's barriers are initialised before any arrival reaches them
  if (kPair) cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0) {
    // ---------------- TMA producer for the token operand (and the LoRA stages)
    // (with debug_stall it loads nothing: no stage completes, the MMA issuer's
    // bounded wait runs out and records a timeout, every role winds down, and
    // no copy or MMA is in flight when the CTA exits)
    if (lane == 0 && !p.debug_stall) {
      int g = 0;
      bool lora_ready = false, stop = false;
      int tile, sb, se;
      for (int idx = 0; !stop && main_piece(p, cta, grid, idx, tile, sb, se); ++idx) {
        const int p0 = feat0(tile);
        const int t0 = (tile / p.p_tiles) * BN + rank * S::kActRows;   // this CTA's token rows
        for (int s = sb; s < se; ++s, ++g) {
          const int slot = g % kMainStages;
          if (!mbar_wait(empty(slot), ((g / kMainStages) & 1) ^ 1, ab)) {
            stop = true;
            break;
          }
          const uint32_t act = base + slot * S::kStageBytes;
          if (s < p.num_kt) {
            mbar_arrive_expect_tx(full(slot), S::kActBytes);
#pragma unroll
            for (int h = 0; h < S::kHalves; ++h)
              tma_load_2d(act + h * (S::kMmaN * 128), &map_act, full(slot), s * kTileK, t0 + h * S::kMmaN);
          } else {
            if (!lora_ready) {
              // the low-rank activations come from the previous kernel: wait for it
              // here (the NF4 stages before this point only read the call's inputs),
              // then let the next kernel start on SMs this grid frees.
              griddep_wait();
              griddep_launch_dependents();
              lora_ready = true;
            }
            int j = s - p.num_kt;
            if (!kTrans && p.grp_n > 0) {
              int g = 0;
              while (g + 1 < p.grp_n && p0 >= p.grp_end[g]) ++g;
              j += g * p.grp_lt0;
            }
            mbar_arrive_expect_tx(full(slot), S::kActBytes + S::kWBytes);
#pragma unroll
            for (int h = 0; h < S::kHalves; ++h)
              tma_load_2d(act + h * (S::kMmaN * 128), &map_lact, full(slot), j * kTileK, t0 + h * S::kMmaN);
            if (kTrans) {
              // A [K, r] rows p0..p0+127, LoRA columns 64j..: K-major
              tma_load_2d(act + S::kActBytes, &map_lw, full(slot), j * kTileK, p0);
            } else {
              // B [r, N] rows 64j.. (the LoRA contraction), columns p0..p0+127: MN-major
              tma_load_2d(act + S::kActBytes, &map_lw, full(slot), p0, j * kTileK);
              tma_load_2d(act + S::kActBytes + 8192, &map_lw, full(slot), p0 + 64, j * kTileK);
            }
          }
        }
      }
      // wait (bounded) until every issued load has landed
      for (int q = g - 1; q >= 0 && q >= g - kMainStages; --q)
        mbar_wait(full(q % kMainStages), (q / kMainStages) & 1, ab, false);
    }
    __syncwarp();
  } else if (warp == 14) {
    // ---------------- TMA producer for the NF4 codes and absmax
    if (lane == 0) {
      int g = 0;
      bool stop = false;
      int tile, sb, se;
      for (int idx = 0; !stop && main_piece(p, cta, grid, idx, tile, sb, se); ++idx) {
        const int p0 = feat0(tile);
        for (int s = sb; s < se; ++s, ++g) {
          const int slot = g % kRaw;
          if (!mbar_wait(raw_empty(slot), ((g / kRaw) & 1) ^ 1, ab)) {
            stop = true;
            break;
          }
          if (s >= p.num_kt) {
            mbar_arrive(raw_full(slot));   // LoRA stage: nothing to load, keep the phases in step
          } else {
            const uint32_t dst = raw_slot(slot);
            mbar_arrive_expect_tx(raw_full(slot), kAbsTma ? (kTrans ? S::kCodeBytes + 1024 : S::kRawBytes)
                                                          : S::kCodeBytes);
            if (!kTrans) {
              tma_load_2d(dst, &map_code, raw_full(slot), 32 * s, p0);                  // W[p0.., 64s..]
              if (kAbsTma) tma_load_2d(dst + S::kCodeBytes, &map_abs, raw_full(slot), s & ~3, p0);
            } else {
              tma_load_2d(dst, &map_code, raw_full(slot), p0 >> 1, 64 * s);             // W[64s.., p0..]
              if (kAbsTma) tma_load_2d(dst + S::kCodeBytes, &map_abs, raw_full(slot), (p0 >> 6) & ~3, 64 * s);
            }
          }
        }
      }
      for (int q = g - 1; q >= 0 && q >= g - kRaw; --q)
        mbar_wait(raw_full(q % kRaw), (q / kRaw) & 1, ab, false);
    }
    __syncwarp();
  } else if (warp == 1 && kPair && rank != 0) {
    // ---------------- odd CTA of a pair: relays "stage in place" to the even CTA,
    // whose thread issues the pair's UMMAs
    if (lane == 0) {
      const uint32_t peer_pfull0 = map_to_cta(pfull(0), 0);
      for (int g = 0; g < g_end; ++g) {
        const int slot = g % kMainStages;
        if (!mbar_wait(full(slot), (g / kMainStages) & 1, ab)) break;
        mbar_arrive_cluster(peer_pfull0 + 8u * slot);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      // A operand majorness: Y -- W tile K-major, B tile MN-major; dX -- W tile MN-major, A tile K-major
      constexpr int kMmaM = kPair ? 2 * kTileP : kTileP;
      constexpr uint32_t idesc_w = umma_idesc_bf16(kMmaM, S::kMmaN, kTrans ? 1 : 0, 0);
      constexpr uint32_t idesc_l = umma_idesc_bf16(kMmaM, S::kMmaN, kTrans ? 0 : 1, 0);
      // descriptors: fixed fields once, the start address (16-byte units) added per MMA
      const uint64_t a_hi_k = sw128_desc(0, 16, 1024), a_hi_mn = sw128_desc(0, 8192, 1024);
      const uint64_t b_hi = sw128_desc(0, 16, 1024);
      const uint32_t base16 = (base & 0x3FFFFu) >> 4;
      // the four K=16 steps of one stage: D (+)= W tile . token tile^T
      auto issue_stage = [&](uint32_t tmem_d, int slot, bool lora, bool first) {
        const bool a_mn = (kTrans != lora);
        const uint64_t a_hi = a_mn ? a_hi_mn : a_hi_k;
        const uint32_t a_step = a_mn ? (2048u >> 4) : (32u >> 4);
        const uint32_t idesc = lora ? idesc_l : idesc_w;
        const uint32_t bs = base16 + static_cast<uint32_t>(slot) * (S::kStageBytes >> 4);
        const uint32_t a0 = bs + (S::kActBytes >> 4);
#pragma unroll
        for (int h = 0; h < S::kHalves; ++h) {
          // token half h (rows h*256..) into accumulator columns h*256..
          const uint32_t b0 = bs + static_cast<uint32_t>(h * S::kMmaN * 128 / 16);
          const uint32_t d = tmem_d + static_cast<uint32_t>(h * S::kMmaN);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = a_hi | (a0 + static_cast<uint32_t>(kk) * a_step);
            const uint64_t bd = b_hi | (b0 + 2u * static_cast<uint32_t>(kk));
            const uint32_t acc_in = (first && kk == 0) ? 0u : 1u;
            if (kPair) umma_bf16_pair(d, ad, bd, idesc, acc_in);
            else umma_bf16(d, ad, bd, idesc, acc_in);
          }
        }
      };
      int g = 0;
      bool ok = true;
      int tile, sb, se;
      for (int idx = 0; ok && main_piece(p, cta, grid, idx, tile, sb, se); ++idx) {
        const int acc = idx % S::kAccs;
        const uint32_t tmem_d = tmem_base + static_cast<uint32_t>(acc * BN);
        const uint32_t te_par = ((idx / S::kAccs) & 1) ^ 1;
        if (!(kPair ? mbar_wait_cluster(tmem_empty(acc), te_par, ab) : mbar_wait(tmem_empty(acc), te_par, ab))) break;
        tc_fence_after_sync();
        int s = sb;
        while (s < se) {
          const int slot = g % kMainStages;
          const uint32_t fpar = (g / kMainStages) & 1;
          if (!mbar_wait(full(slot), fpar, ab) || (kPair && !mbar_wait_cluster(pfull(slot), fpar, ab))) {
            ok = false;
            break;
          }
          // when the next stage of the piece is in place too, issue both at once
          const int slot2 = (g + 1) % kMainStages;
          const uint32_t fpar2 = ((g + 1) / kMainStages) & 1;
          const bool two = (s + 1 < se) && mbar_test_wait(full(slot2), fpar2) &&
                           (!kPair || mbar_test_wait_cluster(pfull(slot2), fpar2));
          tc_fence_after_sync();
          if (kPair) {
            // each stage's commit right behind its own MMAs (a commit completes
            // when all of this thread's earlier MMAs have: committing after the
            // second stage's MMAs frees the first a stage late); the commit
            // frees the stage in both CTAs of the pair.  Measured faster for
            // the pair's deeper ring, slower for the one-CTA form at short stages.
            issue_stage(tmem_d, slot, s >= p.num_kt, s == sb);
            umma_commit_pair(empty(slot), 3);
            if (two) {
              issue_stage(tmem_d, slot2, s + 1 >= p.num_kt, false);
              umma_commit_pair(empty(slot2), 3);
            }
          } else {
            issue_stage(tmem_d, slot, s >= p.num_kt, s == sb);
            if (two) issue_stage(tmem_d, slot2, s + 1 >= p.num_kt, false);
            umma_commit(empty(slot));
            if (two) umma_commit(empty(slot2));
          }
          s += two ? 2 : 1;
          g += two ? 2 : 1;
        }
        if (ok) {
          if (kPair) umma_commit_pair(tmem_full(acc), 3);
          else umma_commit(tmem_full(acc));
        }
      }
      // every MMA issued by this thread has completed once drain_bar flips
      if (kPair) umma_commit_pair(drain_bar, 1);
      else umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, ab, false);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 10) {
    // ---------------- NF4 dequantisation into the UMMA A operand
    const int dw = warp - 2;                  // 0..7
    const int grp = dw >> 2;                  // group g converts stages with g % 2 == grp
    const int i = (dw & 3) * 32 + lane;       // operand row written by this thread
    const uint32_t row_off = static_cast<uint32_t>(i) * 128u;
    const uint32_t swz = static_cast<uint32_t>(i & 7);
    // where this thread's 32 code bytes and absmax sit in a raw slot:
    //   Y : code row i (32 B, 32-B swizzle), absmax row i, column s % 4
    //   dX: code row i % 64 (64 B, 64-B swizzle), bytes 32*(i/64).., absmax row i % 64,
    //       column (p0/64) % 4 + i/64
    uint32_t code_off[2];
    if (!kTrans) {
      const uint32_t x = static_cast<uint32_t>((i >> 2) & 1);
      code_off[0] = static_cast<uint32_t>(i) * 32u + ((0u ^ x) << 4);
      code_off[1] = static_cast<uint32_t>(i) * 32u + ((1u ^ x) << 4);
    } else {
      const uint32_t nl = static_cast<uint32_t>(i & 63), kbl = static_cast<uint32_t>(i >> 6);
      const uint32_t x = (nl >> 1) & 3u;
      code_off[0] = nl * 64u + (((2u * kbl) ^ x) << 4);
      code_off[1] = nl * 64u + (((2u * kbl + 1u) ^ x) << 4);
    }
    const int kblocks = p.K >> 6;
    // absmax straight from global memory when it cannot come by TMA (d_in % 256 != 0)
    auto absmax_direct = [&](int s, int p0) -> float {
      if (kAbsTma || s >= p.num_kt) return 0.0f;
      int n, kb;
      if (!kTrans) {
        n = p0 + i;
        kb = s;
      } else {
        n = s * 64 + (i & 63);
        kb = (p0 >> 6) + (i >> 6);
      }
      if (n >= p.N || kb >= kblocks) return 0.0f;
      return ldg_nc_f32(p.absmax + static_cast<int64_t>(n) * kblocks + kb);
    };
    // this group takes every other stage of the CTA's stage sequence
    StageCursor cur, nxt;
    cur.init(p, cta, grid);
    cur.advance(p, cta, grid, grp);
    nxt = cur;
    nxt.advance(p, cta, grid, 2);
    float am_next = (grp < g_end) ? absmax_direct(cur.s, feat0(cur.tile)) : 0.0f;
    for (int g = grp; g < g_end; g += 2) {
      const int s = cur.s;
      const int p0 = feat0(cur.tile);
      const float am_direct = am_next;
      am_next = (g + 2 < g_end) ? absmax_direct(nxt.s, feat0(nxt.tile)) : 0.0f;
      const int slot = g % kMainStages;
      const uint32_t ph = (g / kMainStages) & 1;
      const int rslot = g % kRaw;
      // every lane acquires the TMA-written codes itself (a shuffle does not order memory)
      if (!__all_sync(0xffffffffu, mbar_wait(raw_full(rslot), (g / kRaw) & 1, ab))) break;
      uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
      float am = am_direct;
      const bool nf4 = s < p.num_kt;
      if (nf4) {
        const uint32_t rs = raw_slot(rslot);
        c0 = ld_shared_v4(rs + code_off[0]);
        c1 = ld_shared_v4(rs + code_off[1]);
        if (kAbsTma) {
          const int col = !kTrans ? (s & 3) : (((p0 >> 6) & 3) + (i >> 6));
          const int row = !kTrans ? i : (i & 63);
          am = ld_shared_f32(rs + S::kCodeBytes + static_cast<uint32_t>(row * 16 + col * 4));
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(empty(slot), ph ^ 1, ab))) break;
      if (nf4) {
        const uint32_t dst = base + slot * S::kStageBytes + S::kActBytes + row_off;
        const Nf4BlockTable tab = nf4_block_table(am);
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) st_shared_v4(dst + ((c ^ swz) << 4), nf4_expand8(words[c], tab));
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full(slot));
      // release the code slot only now: the codes have been consumed, so the loads
      // that read them have completed.  Released right after issuing the loads, the
      // TMA refill of the slot could land before a lane's load had read it.
      if (lane == 0) mbar_arrive(raw_empty(rslot));
      cur = nxt;
      nxt.advance(p, cta, grid, 2);
    }
  } else if (warp >= 10 && warp < 14) {
    // ---------------- epilogue: TMEM -> bf16 -> staging -> TMA store
    // staging: two [32 tokens][64 features] bf16 halves in the 128-B swizzled layout;
    // lanes pair up (shuffle) so each thread stores two adjacent features of one token.
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    const int prow = quarter * 32 + lane;         // output feature within the tile
    // the accumulator's columns may be overwritten: a pair's UMMA issuer (even
    // CTA) waits for the epilogue warps of both CTAs
    const uint32_t te_remote = kPair ? map_to_cta(tmem_empty(0), 0) : 0u;
    auto release_acc = [&](int a) {
      if (kPair) mbar_arrive_cluster(te_remote + 8u * static_cast<uint32_t>(a));
      else mbar_arrive(tmem_empty(a));
    };
    const bool leader = (warp == 10 && lane == 0);
    const uint32_t staging = base + S::kStagingOffset;
    const int f_even = prow & ~1;                 // first of the two features this lane stores
    const uint32_t half_off = static_cast<uint32_t>(f_even >> 6) * 4096u;
    const uint32_t chunk16 = static_cast<uint32_t>((f_even & 63) >> 3);
    const uint32_t in16 = static_cast<uint32_t>((f_even & 7) * 2);
    const bool odd = (lane & 1) != 0;
    // one chunk of 32 tokens x 128 features (this thread: feature prow) -> bf16 -> Y / dX
    auto store_chunk = [&](const float (&f)[32], int p0, int t0, int c0) {
      if (kTrans && p.gate) {
        // dX of the down layer of a SwiGLU block: dh never goes to memory; the
        // gate's backward turns it, with g and u read from gu, into dgu (layout
        // of gu).  dh is rounded to bf16 first, as the unfused block stores it.
        // Lanes pair up (shuffle): the even lane takes tokens 0..15 of the
        // chunk and the odd lane tokens 16..31, each for both features of the
        // pair, so every gu / dgu access is a 4-byte (bf16x2) one, and all 32
        // loads of a lane are issued before the first is used.
        const int n = p0 + f_even;   // the pair's first feature of d_ff
        const bool feat_ok = n < p.K;
        const int64_t pitch = 2 * static_cast<int64_t>(p.K);
        const int64_t gcol = static_cast<int64_t>(n >> 6) * 128 + (n & 63);
        const int tok0 = t0 + c0 + (odd ? 16 : 0);
        float lo[16], hi[16];   // dh of features n and n + 1
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float mine = odd ? f[16 + q] : f[q];
          const float got = __shfl_xor_sync(0xffffffffu, odd ? f[q] : f[16 + q], 1);
          lo[q] = __bfloat162float(__float2bfloat16_rn(odd ? got : mine));
          hi[q] = __bfloat162float(__float2bfloat16_rn(odd ? mine : got));
        }
        uint32_t gw[16], uw[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int tok = tok0 + q;
          const int64_t at = static_cast<int64_t>(tok < p.M ? tok : 0) * pitch + gcol;
          gw[q] = feat_ok ? __ldg(reinterpret_cast<const unsigned int*>(p.gu + at)) : 0u;
          uw[q] = feat_ok ? __ldg(reinterpret_cast<const unsigned int*>(p.gu + at + 64)) : 0u;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int tok = tok0 + q;
          if (!feat_ok || tok >= p.M) continue;
          float dg[2], du[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float gv = __uint_as_float(e ? (gw[q] & 0xFFFF0000u) : (gw[q] << 16));
            const float uv = __uint_as_float(e ? (uw[q] & 0xFFFF0000u) : (uw[q] << 16));
            const float dh = e ? hi[q] : lo[q];
            const float sg = gate_sigmoid(gv);
            du[e] = dh * gv * sg;
            dg[e] = dh * uv * sg * (1.f + gv * (1.f - sg));
          }
          const int64_t at = static_cast<int64_t>(tok) * pitch + gcol;
          *reinterpret_cast<uint32_t*>(p.dgu + at) = pack_bf16x2(dg[0], dg[1]);
          *reinterpret_cast<uint32_t*>(p.dgu + at + 64) = pack_bf16x2(du[0], du[1]);
        }
        return;
      }
      // the previous chunk's store must have read the staging buffer
      if (leader) tma_store_wait_read_all();
      named_bar_sync(1, 128);
#pragma unroll
      for (int jj = 0; jj < kEpiChunk / 2; ++jj) {
        // tokens a and a + 4: their swizzled rows use disjoint bank groups.
        // even lane: token a, features (f, f+1); odd lane: token a+4, features (f-1, f)
        const int a = (jj & 3) + (jj >> 2) * 8;
        const float mine = odd ? f[a + 4] : f[a];
        const float give = odd ? f[a] : f[a + 4];
        const float got = __shfl_xor_sync(0xffffffffu, give, 1);
        const uint32_t pair = odd ? pack_bf16x2(got, mine) : pack_bf16x2(mine, got);
        const uint32_t tok = static_cast<uint32_t>(a + (odd ? 4 : 0));
        st_shared_u32(staging + half_off + tok * 128u + ((chunk16 ^ (tok & 7u)) << 4) + in16, pair);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      // boxes wholly past the last token / feature are not stored
      if (leader && t0 + c0 < p.M && p0 < (kTrans ? p.K : p.N)) {
        tma_store_2d(&map_out, staging, p0, t0 + c0);
        if (p0 + 64 < (kTrans ? p.K : p.N)) tma_store_2d(&map_out, staging + 4096, p0 + 64, t0 + c0);
        tma_store_commit();
      }
      if (!kTrans && p.gate) {
        // Y of the gate/up layer of a SwiGLU block: the staging holds the chunk's
        // gate features (half 0) and the matching up features (half 1), rounded
        // to bf16 as gu stores them; h = silu(g) * u for token a, features
        // 16q .. 16q+15 of the 64, then h through the staging's first half.
        const int et = (warp - 10) * 32 + lane;   // 0..127
        const uint32_t a = static_cast<uint32_t>(et >> 2), q = static_cast<uint32_t>(et & 3);
        uint32_t hw[2][4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t off = a * 128u + (((2u * q + k) ^ (a & 7u)) << 4);
          const uint4 g4v = ld_shared_v4(staging + off), u4v = ld_shared_v4(staging + 4096 + off);
          const uint32_t gw[4] = {g4v.x, g4v.y, g4v.z, g4v.w}, uw[4] = {u4v.x, u4v.y, u4v.z, u4v.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float g0 = __uint_as_float(gw[w] << 16), g1 = __uint_as_float(gw[w] & 0xFFFF0000u);
            const float u0 = __uint_as_float(uw[w] << 16), u1 = __uint_as_float(uw[w] & 0xFFFF0000u);
            hw[k][w] = pack_bf16x2(g0 * gate_sigmoid(g0) * u0, g1 * gate_sigmoid(g1) * u1);
          }
        }
        if (leader) tma_store_wait_read_all();   // the gu stores have read the staging
        named_bar_sync(1, 128);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          st_shared_v4(staging + a * 128u + (((2u * q + k) ^ (a & 7u)) << 4),
                       make_uint4(hw[k][0], hw[k][1], hw[k][2], hw[k][3]));
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader && t0 + c0 < p.M && p0 < p.N) {
          tma_store_2d(&map_h, staging, p0 >> 1, t0 + c0);
          tma_store_commit();
        }
      }
    };
    int tile, sb, se;
    for (int idx = 0; main_piece(p, cta, grid, idx, tile, sb, se); ++idx) {
      const int p0 = feat0(tile);
      const int t0 = (tile / p.p_tiles) * BN;   // all BN tokens: this CTA's TMEM rows hold them
      const int acc = idx % S::kAccs;
      const uint32_t tacc = tmem_base + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(quarter * 32) << 16);
      const uint32_t tf_par = (idx / S::kAccs) & 1;
      if (!__all_sync(0xffffffffu, kPair ? mbar_wait_cluster(tmem_full(acc), tf_par, ab)
                                         : mbar_wait(tmem_full(acc), tf_par, ab)))
        break;
      tc_fence_after_sync();
      if (sb == 0 && se == total) {
        // a whole tile: straight to the output
        for (int c0 = 0; c0 < BN; c0 += kEpiChunk) {
          uint32_t v[32];
          tmem_ld32(tacc + c0, v);
          tmem_ld_wait();
          float f[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) f[q] = __uint_as_float(v[q]);
          store_chunk(f, p0, t0, c0);
        }
        // this accumulator may be overwritten by the MMA of piece idx + 2
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc(acc);
        continue;
      }
      // a piece of a split tile: fp32 partial to this CTA's slot, token-major
      // ([token][feature]) so that each warp store covers 128 contiguous bytes
      const int j = tile - p.dp_tiles;
      float* col = sk_slot<BN, kPair>(p, cta, j, rank) + prow;
      for (int c0 = 0; c0 < BN; c0 += kEpiChunk) {
        uint32_t v[32];
        tmem_ld32(tacc + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) st_global_cg_f32(col + (c0 + q) * kTileP, __uint_as_float(v[q]));
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) release_acc(acc);
      // publish the partial; the last piece of the tile to get here finishes it
      __threadfence();
      named_bar_sync(1, 128);
      const int64_t tile_first = static_cast<int64_t>(j) * total;
      const int c_first = sk_owner(p, tile_first);
      const int c_last = sk_owner(p, tile_first + total - 1);
      if (leader) {
        // the counters were zeroed by the previous kernel
        griddep_wait();
        const int before = atomicAdd(p.counters + (kPair ? 2 * j + rank : j), 1);
        s_last = (before == c_last - c_first) ? 1 : 0;
      }
      named_bar_sync(1, 128);
      if (!s_last) continue;
      __threadfence();
      // contraction order: the CTA holding the first stages comes first
      const float* src_first = sk_slot<BN, kPair>(p, c_first, j, rank) + prow;
      for (int c0 = 0; c0 < BN; c0 += kEpiChunk) {
        float f[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) f[q] = ld_global_cg_f32(src_first + (c0 + q) * kTileP);
        for (int c = c_first + 1; c <= c_last; ++c) {
          const float* src = sk_slot<BN, kPair>(p, c, j, rank) + prow;
#pragma unroll
          for (int q = 0; q < 32; ++q) f[q] += ld_global_cg_f32(src + (c0 + q) * kTileP);
        }
        store_chunk(f, p0, t0, c0);
      }
    }
    if (leader) tma_store_wait_all();
  }

  tc_fence_before_sync();
  __syncthreads();
  // a pair: the even CTA's UMMAs (which read the odd CTA's shared memory and
  // write its TMEM) have completed and no arrival is in flight before either leaves
  if (kPair) cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    if (kPair) tmem_dealloc_pair(tmem_base, S::kAccs * BN);
    else tmem_dealloc(tmem_base, S::kAccs * BN);
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

bool make_map_sw(CUtensorMap* m, CUtensorMapDataType dt, const void* gaddr, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(gaddr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

template <int MODE, int RP, int NSPLIT>
cudaError_t launch_skinny_rp(const CUtensorMap (&maps)[4], const SkinnyParams& sp, int tiles,
                             bool pdl, cudaStream_t stream) {
  constexpr int split = NSPLIT;
  auto kern = lora_skinny_kernel<MODE, RP, NSPLIT>;
  cudaError_t e = set_smem(kern, SkinnySmem<RP>::kBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, split, 1);
  cfg.blockDim = dim3(kSkThreads, 1, 1);
  cfg.dynamicSmemBytes = SkinnySmem<RP>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = split;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  LaunchScope scope(skinny_kind(MODE), stream);
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], sp);
}

template <int MODE, int RP>
cudaError_t launch_skinny_split(const CUtensorMap (&maps)[4], const SkinnyParams& sp, int tiles,
                                int split, bool pdl, cudaStream_t stream) {
  switch (split) {
    case 1: return launch_skinny_rp<MODE, RP, 1>(maps, sp, tiles, pdl, stream);
    case 2: return launch_skinny_rp<MODE, RP, 2>(maps, sp, tiles, pdl, stream);
    case 4: return launch_skinny_rp<MODE, RP, 4>(maps, sp, tiles, pdl, stream);
    default: return launch_skinny_rp<MODE, RP, 8>(maps, sp, tiles, pdl, stream);
  }
}

// `pdl`: launched with programmatic serialisation -- for a kernel whose inputs
// were complete before the previous kernel on the stream started, or one that
// waits for that kernel before it touches global memory (sp.wait_first).
template <int MODE>
cudaError_t launch_skinny(int rp, const CUtensorMap (&maps)[4], const SkinnyParams& sp, int tiles,
                          int split, cudaStream_t stream, bool pdl = false) {
  if (rp == 64) return launch_skinny_split<MODE, 64>(maps, sp, tiles, split, pdl, stream);
  if (rp == 128) return launch_skinny_split<MODE, 128>(maps, sp, tiles, split, pdl, stream);
  return launch_skinny_split<MODE, 256>(maps, sp, tiles, split, pdl, stream);
}

// Split-remainder buffers the main kernel may use (from the workspace).
struct SplitBuffers {
  float* partials;
  size_t partial_bytes;
  int* counters;
  int counter_cap;
};

// Whole tiles for the full waves, then the stages of the remaining tiles
// shared evenly by the units (at least kMinSkStages each), when the buffers
// for the partial tiles are there; otherwise whole tiles only.  A unit is a
// CTA, or a CTA pair (`per_unit` = 2 CTAs, each with its own partial tiles
// and tile counters).  Returns the number of units to launch.
int plan_schedule(int tiles, int total, int bn, const SplitBuffers& sb, MainParams& mp, int sms,
                  int per_unit = 1) {
  const int full = tiles / sms, rem = tiles % sms;
  mp.sk_tiles = 0;
  mp.sk_ctas = 0;
  if (rem != 0 && sb.partials != nullptr && sb.counters != nullptr) {
    const int64_t len = static_cast<int64_t>(rem) * total;
    // never fewer CTAs than remaining tiles (that would be worse than whole tiles)
    const int ctas = static_cast<int>(std::min<int64_t>(sms, std::max<int64_t>(rem, len / kMinSkStages)));
    const size_t need = static_cast<size_t>(2) * ctas * per_unit * kTileP * bn * sizeof(float);
    if (need <= sb.partial_bytes && rem * per_unit <= sb.counter_cap) {
      mp.dp_tiles = full * sms;
      mp.dp_rounds = full;
      mp.sk_tiles = rem;
      mp.sk_ctas = ctas;
      mp.partials = sb.partials;
      mp.counters = sb.counters;
      return full > 0 ? sms : ctas;
    }
  }
  const int grid = std::min(tiles, sms);
  mp.dp_tiles = tiles;
  mp.dp_rounds = (tiles + grid - 1) / grid;
  mp.partials = nullptr;
  mp.counters = nullptr;
  return grid;
}

template <int BN, bool kTrans, bool kAbsTma, bool kPair>
cudaError_t launch_main_bn(const CUtensorMap (&maps)[7], MainParams mp, int P, int M, const SplitBuffers& sb,
                           cudaStream_t stream) {
  using S = MainSmem<BN, kPair>;
  auto kern = lora_main_kernel<BN, kTrans, kAbsTma, kPair>;
  cudaError_t e = set_smem(kern, S::kBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kMainThreads, 1, 1);
  cfg.dynamicSmemBytes = S::kBytes;
  cfg.stream = stream;
  // programmatic serialisation: the NF4 stages start while the low-rank kernel
  // before this one finishes; the producer waits for it before the LoRA stages
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kPair ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kPair ? 2 : 1;
  // units: one CTA per SM, or as many CTA pairs as can be resident at once
  int units = sm_count();
  if (kPair) {
    // queried once (thread-safe initialisation); 0 if the query failed
    static const int pairs = [&]() {
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2 * (units / 2), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess) return 0;
      return std::max(1, std::min(n, units / 2));
    }();
    if (pairs == 0) return cudaErrorInvalidConfiguration;
    units = pairs;
  }
  mp.p_tiles = (P + (kPair ? 2 * kTileP : kTileP) - 1) / (kPair ? 2 * kTileP : kTileP);
  mp.t_tiles = (M + BN - 1) / BN;
  const int grid = plan_schedule(mp.p_tiles * mp.t_tiles, mp.num_kt + mp.num_lt, BN, sb, mp, units, kPair ? 2 : 1);
  cfg.gridDim = dim3(grid * (kPair ? 2 : 1), 1, 1);
  LaunchScope scope(kTrans ? kKindMainDx : kKindMainFwd, stream);
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], mp);
}

template <int BN, bool kTrans, bool kPair = false>
cudaError_t launch_main_abs(const CUtensorMap (&maps)[7], const MainParams& mp, bool abs_tma, int P,
                            int M, const SplitBuffers& sb, cudaStream_t stream) {
  if (abs_tma) return launch_main_bn<BN, kTrans, true, kPair>(maps, mp, P, M, sb, stream);
  return launch_main_bn<BN, kTrans, false, kPair>(maps, mp, P, M, sb, stream);
}

int pick_bn(int M) { return M <= 32 ? 32 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256)); }

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
                        const float* absmax, const Workspace& ws, int* status, cudaStream_t stream,
                        const GateIo& gate = GateIo{}) {
  const int P = kTrans ? d.K : d.N;     // output features
  const int C = kTrans ? d.N : d.K;     // contraction length of the NF4 part
  const int bn = pick_bn(d.M);
  const bool abs_tma = (d.K % 256) == 0;   // absmax rows are 16-byte multiples
  // CTA pairs for the widest token tiles; the two CTAs of a pair share the
  // low-rank contraction, so stacked projections need group ends on 256-row bounds
  bool pair = bn == 256 && P >= 2 * kTileP;
  if (!kTrans && d.groups.n > 0)
    for (int g = 0; g < d.groups.n; ++g) pair = pair && d.groups.end[g] % (2 * kTileP) == 0;
  CUtensorMap maps[7];
  const bool gated = kTrans ? gate.dgu != nullptr : gate.h != nullptr;
  if (kTrans && gated) out = gate.dgu;   // dX is not stored; its map is never used
  const int box_t = pair ? bn / 2 : (bn < 256 ? bn : 256);   // token rows per TMA box
  bool ok = map_bf16(&maps[0], act, C, d.M, 64, box_t, true) && map_bf16(&maps[1], lact, d.rp, d.M, 64, box_t, true) &&
            make_map(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, P, d.M, static_cast<uint64_t>(P) * 2, 64,
                     kEpiChunk, true);
  if (kTrans) ok = ok && map_bf16(&maps[2], lw, lw_cols, d.K, 64, kTileP, true);   // A [K, r]
  else ok = ok && map_bf16(&maps[2], lw, d.N, d.r, 64, 64, true);                   // B [r, N]
  // NF4 codes as bytes [N, K/2]; absmax as fp32 [N, K/64]
  ok = ok && make_map_sw(&maps[4], CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, d.K / 2, d.N, d.K / 2,
                         kTrans ? 64 : 32, kTrans ? 64 : kTileP,
                         kTrans ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  if (abs_tma)
    ok = ok && make_map_sw(&maps[5], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, absmax, d.K / 64, d.N, d.K / 16, 4,
                           kTrans ? 64 : kTileP, CU_TENSOR_MAP_SWIZZLE_NONE);
  else
    maps[5] = maps[4];
  if (!kTrans && gated)   // h [M, N/2]
    ok = ok && make_map(&maps[6], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, gate.h, d.N / 2, d.M,
                        static_cast<uint64_t>(d.N / 2) * 2, 64, kEpiChunk, true);
  else
    maps[6] = maps[3];
  if (!ok) return cudaErrorInvalidValue;
  MainParams mp;
  mp.gate = gated ? 1 : 0;
  mp.gu = gate.gu;
  mp.dgu = gate.dgu;
  mp.absmax = absmax;
  mp.M = d.M;
  mp.K = d.K;
  mp.N = d.N;
  mp.num_kt = (C + kTileK - 1) / kTileK;
  mp.num_lt = d.rp / kTileK;
  mp.grp_n = 0;
  mp.grp_lt0 = 0;
  if (!kTrans && d.groups.n > 0) {
    mp.grp_n = d.groups.n;
    mp.grp_lt0 = d.groups.width / kTileK;
    mp.num_lt = mp.grp_lt0;
    for (int g = 0; g < kMaxLoraGroups; ++g) mp.grp_end[g] = d.groups.end[g];
  }
  mp.debug_stall = take_debug_stall() ? 1 : 0;
  mp.status = status;
  const SplitBuffers sb = {ws.partials, ws.partial_bytes, ws.counters, ws.counter_cap};
  if (bn == 32) return launch_main_abs<32, kTrans>(maps, mp, abs_tma, P, d.M, sb, stream);
  if (bn == 64) return launch_main_abs<64, kTrans>(maps, mp, abs_tma, P, d.M, sb, stream);
  if (bn == 128) return launch_main_abs<128, kTrans>(maps, mp, abs_tma, P, d.M, sb, stream);
  if (pair) return launch_main_abs<256, kTrans, true>(maps, mp, abs_tma, P, d.M, sb, stream);
  return launch_main_abs<256, kTrans>(maps, mp, abs_tma, P, d.M, sb, stream);
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

// Workspace: padded A [K, rp], bf16(s*T) and bf16(s*G) [M, rp], then the
// counters (split tiles of the main kernel, or panels of the token-stream
// kernel) and the partial tiles (two per SM).
bool make_bf16_map_sw128(CUtensorMap* m, const void* gaddr, uint64_t cols, uint64_t rows, uint32_t box_cols,
                         uint32_t box_rows) {
  return map_bf16(m, gaddr, cols, rows, box_cols, box_rows, true);
}

bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* gaddr, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  return make_map_sw(m, dt, gaddr, inner, outer, row_bytes, box_inner, box_outer, sw);
}

size_t split_partial_bytes(const LayerDims& d) {
  const int sms = sm_count();
  const size_t main_bytes = static_cast<size_t>(2) * sms * kTileP * pick_bn(d.M) * sizeof(float);
  if (d.M > kStreamMaxTokens) return main_bytes;
  return std::max(main_bytes, stream_partial_bytes(d, sms));
}

int counter_slots(const LayerDims& d) { return std::max(sm_count(), stream_counter_slots(d)); }

size_t workspace_bytes(const LayerDims& d) {
  const size_t rp = static_cast<size_t>(d.rp);
  return align_up(static_cast<size_t>(d.K) * rp * 2) + 2 * align_up(static_cast<size_t>(d.M) * rp * 2) +
         align_up(static_cast<size_t>(counter_slots(d)) * sizeof(int)) + align_up(split_partial_bytes(d));
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
  b += align_up(static_cast<size_t>(d.M) * rp * 2);
  w.counters = reinterpret_cast<int*>(b);
  w.counter_cap = counter_slots(d);
  b += align_up(static_cast<size_t>(w.counter_cap) * sizeof(int));
  w.partials = reinterpret_cast<float*>(b);
  w.partial_bytes = split_partial_bytes(d);
  return w;
}

cudaError_t run_forward(const LayerDims& d, const uint16_t* X, const uint8_t* packed,
                        const float* absmax, const uint16_t* A, const uint16_t* B, uint16_t* Y,
                        float* XA, const Workspace& ws, int* status, cudaStream_t stream, uint16_t* gate_h) {
  cudaError_t e = launch_pad_a(d, A, ws, stream);
  if (e != cudaSuccess) return e;
  const LowRankA la = low_rank_a(d, A, ws);
  const int sms = sm_count();
  if (stream_applies(d, ws, sms)) {
    // 1..16 tokens: T on one small cluster beside the weight stream
    e = launch_xa_small(d, X, la.ptr, la.cols, XA, ws, status, stream);
    if (e == cudaSuccess) e = launch_stream_fwd(d, X, packed, absmax, B, ws, Y, status, sms, stream);
    // the token-stream kernel's 16-row groups hold gate or up features, never
    // both: the gate runs as its own pass over the interleaved output
    if (e == cudaSuccess && gate_h != nullptr) e = launch_swiglu_fwd(Y, d.M, d.N / 2, gate_h, true, stream);
    return e;
  }
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
    sp.zero = ws.counters;
    sp.n_zero = ws.counters != nullptr ? ws.counter_cap : 0;
    sp.status = status;
    const int tiles = sp.job[0].tiles;
    sp.wait_first = 1;
    e = launch_skinny<kRowsT>(d.rp, maps, sp, tiles, pick_split(tiles, sp.num_ct), stream, true);
    if (e != cudaSuccess) return e;
  }
  GateIo gate;
  gate.h = gate_h;
  return launch_main<false>(d, X, ws.s_t, B, d.r, Y, packed, absmax, ws, status, stream, gate);
}

cudaError_t run_backward(const LayerDims& d, const uint16_t* X, const uint16_t* dY,
                         const uint8_t* packed, const float* absmax, const uint16_t* A,
                         const uint16_t* B, const float* XA, uint16_t* dX, float* dA, float* dB,
                         const Workspace& ws, int* status, cudaStream_t stream, const uint16_t* gate_gu,
                         uint16_t* gate_dgu) {
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
    sp.zero = ws.counters;
    sp.n_zero = ws.counters != nullptr ? ws.counter_cap : 0;
    sp.status = status;
    const int tiles = sp.job[0].tiles;
    sp.wait_first = 1;
    e = launch_skinny<kRowsG>(d.rp, maps, sp, tiles, pick_split(tiles, sp.num_ct), stream, true);
    if (e != cudaSuccess) return e;
  }
  // dX first; the dA/dB kernel then runs in the SMs dX's last tiles leave idle.  It may start
  // before dX finishes because dX lets it go only after its own wait on the G kernel.
  const bool with_dx = dX != nullptr || gate_dgu != nullptr;
  if (with_dx) {
    GateIo gate;
    gate.gu = gate_gu;
    gate.dgu = gate_dgu;
    e = launch_main<true>(d, dY, ws.s_g, la.ptr, la.cols, dX, packed, absmax, ws, status, stream, gate);
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
    if (d.groups.n > 0) {
      // stacked projections: dB only in the diagonal blocks
      sp.grp_n = d.groups.n;
      sp.grp_width = d.groups.width;
      for (int g = 0; g < kMaxLoraGroups; ++g) sp.grp_end[g] = d.groups.end[g];
    }
    sp.job[1].rows = d.N;
    sp.job[1].tiles = (d.N + kTileP - 1) / kTileP;
    sp.job[1].out_f32 = dB;
    sp.status = status;
    const int tiles = sp.job[0].tiles + sp.job[1].tiles;
    e = launch_skinny<kRed>(d.rp, maps, sp, tiles, pick_split(tiles, sp.num_ct), stream, with_dx);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace qlora
