// lora_stream.cu -- the forward Y = X . W_deq^T + s . (X . A) . B for a handful of
// tokens (M <= 16), where the layer is a stream of its NF4 weight.
//
// Operation: the fused QLoRA linear of the Unsloth pages ("UnSloth加速原理：CUDA内核
// 融合与内存优化", section "内核融合"; "这不是“魔法”是把Unsloth的底层优化逻辑榨干了用",
// section 1), the same result as the main kernel.  With so few tokens the work is
// 0.5625 bytes of codes and absmax per weight element against 2*M flops, so the
// kernel is built around moving the weight once at the HBM rate:
//
//   * Work unit: a stage of 64 weight rows x 256 input features (four NF4
//     blocks).  The flattened list of stages (panel-major) is split evenly over
//     one CTA per SM.  A producer warp streams a CTA's stages through a ring of
//     shared-memory slots with TMA (codes, absmax, and the matching columns of
//     X), several stages ahead; sixteen consumer warps each take 32 features
//     of every stage for 32 of its 64 rows.  With at least as many 64-row
//     panels as CTAs each CTA takes whole panels (at most one panel of
//     imbalance, and no partial sums between CTAs); with fewer, the stages are
//     split evenly and a panel may be shared by CTAs.
//   * Every consumer thread decodes its share of the codes straight into the
//     register operands of mma.sync (m16n8k16, bf16 -> fp32): one shared-memory
//     lookup per code byte in a 256-entry table of bf16 code pairs (one copy per
//     lane, so lookups never conflict).  The dequantised weight never goes back
//     to shared memory or to the tensor memory, which a tcgen05 operand would
//     need: here the shared-memory pipe, not the tensor core, sets the pace, and
//     a tcgen05 MMA would double its traffic.
//   * The block scale is applied after the block's MMAs: D = sum over the
//     warp's 32 features of bf16(level[q]) * x, then acc += absmax * D in fp32.
//     This is the sum of bf16(level[q] * absmax) * x up to the rounding of the
//     weight (both within 2^-9 of the exact level * absmax).
//   * The contraction order inside an MMA is free: thread (g, c) of the MMA
//     takes 8 consecutive features (one 32-bit word of codes per row) and the
//     activations are read in the same permuted order.
//   * The decode table is a compile-time array in global memory, copied into
//     shared memory by one bulk copy while the first stages load.
//   * At the end of a panel segment the consumers leave their partials in
//     shared memory and go on; four epilogue warps (one per 16-row group) sum
//     them, add the low-rank term s*T.B when the CTA holds the panel's first
//     stage (B and bf16(s*T) copied in with cp.async, multiplied with
//     ldmatrix.trans + mma), and write the panel, overlapping the next
//     segment's stages.
//   * A panel split between CTAs is finished by the last of them to arrive (a
//     counter per panel, zeroed by the rank-r kernel that runs before this one):
//     it adds the fp32 partials in CTA order, so the result does not depend on
//     timing.
//
// Every mbarrier wait is bounded (kWaitLimitNs): on expiry the CTA records a
// timeout in the status word and winds down.

#include <cuda_bf16.h>
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "nf4_lut.cuh"
#include "ptx.cuh"

namespace qlora {
namespace {

constexpr int kSlices = 8;                         // 32-feature slices of a stage
constexpr int kConsumerWarps = 2 * kSlices;        // each slice for the upper and the lower 32 rows
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarps = 4;                  // one per 16-row group of a panel
constexpr int kEpilogueWarp0 = kConsumerWarps + 1;
constexpr int kEpilogueThreads = kEpilogueWarps * 32;
constexpr int kStreamThreads = kConsumers + 32 + kEpilogueThreads;
constexpr int kPanelRows = 64;                     // weight rows per panel (4 MMA row groups)
constexpr int kStageK = 256;                       // input features per stage (4 NF4 blocks)
constexpr int kSlotStride = kPanelRows + 4;        // fp32 per token row of a warp's panel partial
constexpr int kSlotFloats = 16 * kSlotStride;      // up to 16 tokens
constexpr int kPartialFloats = 16 * kPanelRows;    // one panel partial in global memory
constexpr int kLutWords = 256 * 32;                // 256 code bytes x 32 lane copies
constexpr int kBsStride = 64 * 2 + 16;             // bytes per rank row of the panel's B columns
constexpr int kTsStride = 128 * 2 + 16;            // bytes per token row of bf16(s*T)
constexpr int kEpiBar = 1;                         // epilogue-warps-only barrier

// bf16 bit patterns (round to nearest even) of the NF4 levels, in code order:
// the host copy kNF4LevelsHost rounded; launch_stream_fwd checks the two agree.
constexpr uint16_t kLevelBf16[16] = {0xBF80, 0xBF32, 0xBF06, 0xBECA, 0xBE92, 0xBE3D, 0xBDBA, 0x0000,
                                     0x3DA3, 0x3E25, 0x3E7C, 0x3EAD, 0x3EE2, 0x3F10, 0x3F39, 0x3F80};

// The decode table: word 32 * v + l (l = lane copy) holds, for code byte v,
// bf16(level[v >> 4]) (the byte's first element) in the low half and
// bf16(level[v & 15]) in the high half.
struct alignas(16) PairTable {
  uint32_t w[kLutWords];
};

constexpr PairTable make_pair_table() {
  PairTable t{};
  for (int i = 0; i < kLutWords; ++i) {
    const int v = i >> 5;
    t.w[i] = static_cast<uint32_t>(kLevelBf16[v >> 4]) | (static_cast<uint32_t>(kLevelBf16[v & 15]) << 16);
  }
  return t;
}

__device__ const PairTable g_pair_table = make_pair_table();

// Shared memory: the ring (1024-aligned for the 128-byte swizzle), then the
// decode table, the warps' panel partials, the low-rank operands, the barriers.
template <int MT>
struct StreamSmem {
  static constexpr int kCodeBytes = kPanelRows * 128;            // [64 rows][128 B], swizzled
  static constexpr int kXBoxBytes = MT * 8 * 128;                // [8*MT tokens][64 features]
  static constexpr int kAbsOffset = kCodeBytes + 4 * kXBoxBytes; // [64 rows][4 blocks] fp32
  static constexpr int kStageBytes = kAbsOffset + kPanelRows * 16;
  static constexpr int kStages = MT == 1 ? 8 : 6;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kLutOffset = kRingBytes;
  static constexpr int kSlotOffset = kLutOffset + kLutWords * 4;
  static constexpr int kBsOffset = kSlotOffset + kSlices * kSlotFloats * 4;
  static constexpr int kTsOffset = kBsOffset + 128 * kBsStride;
  static constexpr int kBarOffset = kTsOffset + 16 * kTsStride;
  static constexpr int kBytes = kBarOffset + 16 * kStages + 32 + 1024;   // + table/slot barriers, slack
  static_assert(kStageBytes % 1024 == 0, "stages keep the swizzle alignment");
  static_assert(kBytes <= 227 * 1024, "fits the shared memory of one CTA");
};

struct StreamParams {
  const uint16_t* B;        // [r, N] bf16
  const uint16_t* s_t;      // [M, rp] bf16(s*T), zero columns r..rp-1
  uint16_t* Y;              // [M, N] bf16
  float* partials;          // [2 * gridDim.x][16 * 64]
  int* counters;            // [panels]
  int* status;
  int M, N, r, rp;
  int units;                // stages per panel: K / 256
  long long total;          // panels * units
  int whole;                // 1: every CTA takes whole panels (panels >= CTAs)
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// 16-byte asynchronous copy global -> shared; src_bytes 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Four 8x8 bf16 matrices from shared memory, transposed (the A operand of an
// m16n8k16 MMA from a [k][m] row-major tile).
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&a)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr)
               : "memory");
}

// D += A . B for one m16n8k16 tile, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte i of a code word through the lane's copy of the pair table: the copy
// for code byte v and lane l sits at byte offset 128 * v + 4 * l.
template <int I>
__device__ __forceinline__ uint32_t lut_pair(const uint8_t* lut, uint32_t lane4, uint32_t w) {
  const uint32_t off = ((I == 0 ? (w << 7) : (w >> (8 * I - 7))) & 0x7F80u) | lane4;
  return *reinterpret_cast<const uint32_t*>(lut + off);
}

// One consumer warp's share of a stage: features 32*kw .. +31 of the stage for
// row groups 2*gh and 2*gh + 1 (rows 32*gh .. +31).  Thread (g4 = lane/4,
// c = lane%4) holds MMA rows g4 and g4 + 8 of each row group and features
// 8c .. 8c+7 of the warp's 32.  Plain shared-memory loads (ordered after the
// stage's barrier wait by its memory clobber), so the compiler can interleave
// the independent row groups.
template <int MT>
__device__ __forceinline__ void consume_stage(const uint8_t* st, const uint8_t* lut, uint32_t lane4, int kw, int gh,
                                              int g4, int c, float (&acc)[2][MT][4]) {
  using S = StreamSmem<MT>;
  uint4 xv[MT];
#pragma unroll
  for (int j = 0; j < MT; ++j) {
    const int tok = 8 * j + g4;
    const int ch = 4 * (kw & 1) + c;
    xv[j] = *reinterpret_cast<const uint4*>(st + S::kCodeBytes + (kw >> 1) * S::kXBoxBytes + tok * 128 +
                                            ((ch ^ (tok & 7)) << 4));
  }
  const int code_col = ((kw ^ g4) << 4) + 4 * c;   // row & 7 == g4
  uint32_t wa[2], wb[2];
  float sa[2], sb[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int ra = 16 * (2 * gh + h) + g4, rb = ra + 8;
    wa[h] = *reinterpret_cast<const uint32_t*>(st + ra * 128 + code_col);
    wb[h] = *reinterpret_cast<const uint32_t*>(st + rb * 128 + code_col);
    sa[h] = *reinterpret_cast<const float*>(st + S::kAbsOffset + ra * 16 + (kw >> 1) * 4);
    sb[h] = *reinterpret_cast<const float*>(st + S::kAbsOffset + rb * 16 + (kw >> 1) * 4);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    // step 0 covers features 8c .. 8c+3 (code bytes 0, 1), step 1 features 8c+4 .. +7
    const uint32_t a0[4] = {lut_pair<0>(lut, lane4, wa[h]), lut_pair<0>(lut, lane4, wb[h]),
                            lut_pair<1>(lut, lane4, wa[h]), lut_pair<1>(lut, lane4, wb[h])};
    const uint32_t a1[4] = {lut_pair<2>(lut, lane4, wa[h]), lut_pair<2>(lut, lane4, wb[h]),
                            lut_pair<3>(lut, lane4, wa[h]), lut_pair<3>(lut, lane4, wb[h])};
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(d, a0, xv[j].x, xv[j].y);
      mma_16816(d, a1, xv[j].z, xv[j].w);
      acc[h][j][0] = fmaf(sa[h], d[0], acc[h][j][0]);
      acc[h][j][1] = fmaf(sa[h], d[1], acc[h][j][1]);
      acc[h][j][2] = fmaf(sb[h], d[2], acc[h][j][2]);
      acc[h][j][3] = fmaf(sb[h], d[3], acc[h][j][3]);
    }
  }
}

// The panel's B columns [rp][64] -> shared memory, by the epilogue warps (et = 0..127).
__device__ __forceinline__ void stage_lowrank_b(const StreamParams& p, int n0, uint32_t bs, int et) {
  for (int e = et; e < p.rp * 8; e += kEpilogueThreads) {
    const int j = e >> 3, q = e & 7, n = n0 + 8 * q;
    const bool ok = j < p.r && n < p.N;
    cp_async16(bs + j * kBsStride + q * 16,
               ok ? static_cast<const void*>(p.B + static_cast<int64_t>(j) * p.N + n) : p.B, ok ? 16u : 0u);
  }
  cp_async_commit();
}

// bf16(s*T) [8*MT tokens][rp] -> shared memory, by the epilogue warps (after
// they wait for the kernel that writes it).
template <int MT>
__device__ __forceinline__ void stage_lowrank_t(const StreamParams& p, uint32_t ts, int et) {
  const int chunks = p.rp / 8;
  for (int e = et; e < MT * 8 * chunks; e += kEpilogueThreads) {
    const int tok = e / chunks, q = e % chunks;
    const bool ok = tok < p.M;
    cp_async16(ts + tok * kTsStride + q * 16,
               ok ? static_cast<const void*>(p.s_t + static_cast<int64_t>(tok) * p.rp + 8 * q) : p.s_t,
               ok ? 16u : 0u);
  }
  cp_async_commit();
}

__device__ __forceinline__ int owner_cta(long long x, long long total, int G) {
  return static_cast<int>(((x + 1) * G - 1) / total);
}

template <int MT>
__global__ void __launch_bounds__(kStreamThreads, 1)
    lora_stream_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_abs,
                       const __grid_constant__ CUtensorMap map_x, const StreamParams p) {
  using S = StreamSmem<MT>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_last, s_abort;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t bar_full = base + S::kBarOffset, bar_empty = bar_full + 8 * S::kStages;
  const uint32_t bar_table = bar_empty + 8 * S::kStages;
  const uint32_t bar_slots_full = bar_table + 8, bar_slots_free = bar_table + 16;
  float* const slots = reinterpret_cast<float*>(gbase + S::kSlotOffset);

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  // whole panels when there are at least as many panels as CTAs (no panel is
  // split, so no partials); otherwise the stages are split evenly
  const long long panels = p.total / p.units;
  const long long u_begin = p.whole ? panels * cta / G * p.units : p.total * cta / G;
  const long long u_end = p.whole ? panels * (cta + 1) / G * p.units : p.total * (cta + 1) / G;
  const int n_stages = static_cast<int>(u_end - u_begin);
  Abort ab{&s_abort, p.status};

  if (t == 0) {
    s_abort = 0;
    for (int i = 0; i < S::kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kConsumerWarps);
    }
    mbar_init(bar_table, 1);
    mbar_init(bar_slots_full, kConsumerWarps);
    mbar_init(bar_slots_free, kEpilogueWarps);
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---- producer: the decode table, then codes, absmax and X columns of each
    //      stage, kStages ahead
    if (lane == 0) {
      const uint32_t table = base + S::kLutOffset;
      mbar_arrive_expect_tx(bar_table, kLutWords * 4);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        bulk_load_1d(table + q * (kLutWords / 4) * 4, g_pair_table.w + q * (kLutWords / 4), kLutWords, bar_table);
      tma_prefetch_map(&map_codes);
      tma_prefetch_map(&map_abs);
      tma_prefetch_map(&map_x);
      int i = 0;
      for (; i < n_stages; ++i) {
        const int slot = i % S::kStages;
        const uint32_t ph = (i / S::kStages) & 1;
        if (!mbar_wait(bar_empty + 8 * slot, ph ^ 1, ab)) break;
        const long long u = u_begin + i;
        const int panel = static_cast<int>(u / p.units), q = static_cast<int>(u % p.units);
        const uint32_t st = base + slot * S::kStageBytes, full = bar_full + 8 * slot;
        mbar_arrive_expect_tx(full, S::kStageBytes);
        tma_load_2d(st, &map_codes, full, q * 128, panel * kPanelRows);
#pragma unroll
        for (int b = 0; b < 4; ++b)
          tma_load_2d(st + S::kCodeBytes + b * S::kXBoxBytes, &map_x, full, q * kStageK + 64 * b, 0);
        tma_load_2d(st + S::kAbsOffset, &map_abs, full, q * 4, panel * kPanelRows);
      }
      // no copy may still be landing when the CTA exits
      mbar_wait(bar_table, 0, ab, false);
      for (int k = i - 1; k >= 0 && k >= i - S::kStages; --k)
        mbar_wait(bar_full + 8 * (k % S::kStages), (k / S::kStages) & 1, ab, false);
    }
    return;
  }

  const int g4 = lane >> 2, c = lane & 3;

  if (warp >= kEpilogueWarp0) {
    // ---- epilogue: warp ew takes row group ew of every panel segment, behind the consumers
    const int ew = warp - kEpilogueWarp0, et = t - kEpilogueWarp0 * 32;
    const uint32_t bs = base + S::kBsOffset, ts = base + S::kTsOffset;
    const int first_panel = static_cast<int>(u_begin / p.units);
    bool waited = false;
    int k = 0;   // segment index within the CTA
    for (long long seg = u_begin; seg < u_end; ++k) {
      const int panel = static_cast<int>(seg / p.units);
      const long long pu0 = static_cast<long long>(panel) * p.units;
      const long long seg_end = u_end < pu0 + p.units ? u_end : pu0 + p.units;
      const int n0 = panel * kPanelRows;
      const bool lowrank = seg == pu0;   // this CTA holds the panel's first stage
      if (lowrank) {
        stage_lowrank_b(p, n0, bs, et);
        if (!waited) {
          griddep_wait();   // bf16(s*T) and the counters come from the kernel before this one
          waited = true;
        }
        stage_lowrank_t<MT>(p, ts, et);
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_slots_full, k & 1, ab));
      // the eight slices' partials of this warp's 16 rows
      float acc[MT][4];
#pragma unroll
      for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int at = (8 * j + 2 * c + (e & 1)) * kSlotStride + 16 * ew + g4 + 8 * (e >> 1);
          float sum = 0.f;
#pragma unroll
          for (int b = 0; b < kSlices; ++b) sum += slots[b * kSlotFloats + at];
          acc[j][e] = sum;
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_slots_free);   // the consumers may write the next segment's partials
      if (lowrank) {
        cp_async_wait_all();
        named_bar_sync(kEpiBar, kEpilogueThreads);   // every copy of B and bf16(s*T) has landed
        const int mi = lane >> 3, rr = lane & 7;
        for (int ks = 0; ks < p.rp / 16; ++ks) {
          uint32_t a[4];
          ldmatrix_x4_trans(a, bs + (16 * ks + rr + ((mi & 2) ? 8 : 0)) * kBsStride +
                                   (16 * ew + ((mi & 1) ? 8 : 0)) * 2);
#pragma unroll
          for (int j = 0; j < MT; ++j) {
            const uint32_t row = ts + (8 * j + g4) * kTsStride + (16 * ks + 2 * c) * 2;
            mma_16816(acc[j], a, lds32(row), lds32(row + 16));
          }
        }
      }
      const int first_c = p.whole ? cta : owner_cta(pu0, p.total, G);
      const int last_c = p.whole ? cta : owner_cta(pu0 + p.units - 1, p.total, G);
      if (first_c == last_c) {
        // the whole panel is this CTA's
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = 8 * j + 2 * c + (e & 1), n = n0 + 16 * ew + g4 + 8 * (e >> 1);
            if (ok && tok < p.M && n < p.N)
              p.Y[static_cast<int64_t>(tok) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j][e]));
          }
      } else {
        const int my_slot = 2 * cta + (panel == first_panel ? 0 : 1);
        float* part = p.partials + static_cast<int64_t>(my_slot) * kPartialFloats;
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            __stcg(part + (8 * j + 2 * c + (e & 1)) * kPanelRows + 16 * ew + g4 + 8 * (e >> 1), acc[j][e]);
        __threadfence();
        named_bar_sync(kEpiBar, kEpilogueThreads);
        if (et == 0) {
          if (!waited) griddep_wait();   // the counters are zeroed by the kernel before this one
          __threadfence();
          const int arrived = atomicAdd(p.counters + panel, 1);
          s_last = (ok && arrived == last_c - first_c) ? 1 : 0;
          if (s_last) __threadfence();
        }
        waited = true;
        named_bar_sync(kEpiBar, kEpilogueThreads);
        if (s_last) {
          // the last CTA to finish a piece of this panel adds the pieces in CTA order
#pragma unroll
          for (int j = 0; j < MT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = 8 * j + 2 * c + (e & 1), row = 16 * ew + g4 + 8 * (e >> 1);
              float sum = 0.f;
              for (int q = first_c; q <= last_c; ++q) {
                const long long q_begin = p.total * q / G;
                const int q_slot = 2 * q + (static_cast<int>(q_begin / p.units) == panel ? 0 : 1);
                sum += __ldcg(p.partials + static_cast<int64_t>(q_slot) * kPartialFloats + tok * kPanelRows + row);
              }
              if (tok < p.M && n0 + row < p.N)
                p.Y[static_cast<int64_t>(tok) * p.N + n0 + row] = __bfloat16_as_ushort(__float2bfloat16_rn(sum));
            }
        }
      }
      named_bar_sync(kEpiBar, kEpilogueThreads);   // B, bf16(s*T) and s_last are reused by the next segment
      seg = seg_end;
    }
    return;
  }

  // ---- consumers
  const uint8_t* const lut_b = gbase + S::kLutOffset;
  const uint32_t lane4 = static_cast<uint32_t>(lane) * 4u;
  const int kw = warp % kSlices, gh = warp / kSlices;
  mbar_wait(bar_table, 0, ab);   // the decode table has landed
  int i = 0;   // stage index within the CTA's range
  int k = 0;   // segment index
  for (long long seg = u_begin; seg < u_end; ++k) {
    const int panel = static_cast<int>(seg / p.units);
    const long long pu0 = static_cast<long long>(panel) * p.units;
    const long long seg_end = u_end < pu0 + p.units ? u_end : pu0 + p.units;

    float acc[2][MT][4];
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][j][e] = 0.f;

    for (long long u = seg; u < seg_end; ++u, ++i) {
      const int slot = i % S::kStages;
      const uint32_t ph = (i / S::kStages) & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_full + 8 * slot, ph, ab));
      if (ok) consume_stage<MT>(gbase + slot * S::kStageBytes, lut_b, lane4, kw, gh, g4, c, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
    }

    // the warp's rows of its slice's partial panel -> shared memory, [token][row],
    // once the epilogue has taken the previous segment's
    if (k > 0) __all_sync(0xffffffffu, mbar_wait(bar_slots_free, (k - 1) & 1, ab));
    float* slot = slots + kw * kSlotFloats;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const int row = 16 * (2 * gh + h) + g4, tok = 8 * j + 2 * c;
        slot[tok * kSlotStride + row] = acc[h][j][0];
        slot[(tok + 1) * kSlotStride + row] = acc[h][j][1];
        slot[tok * kSlotStride + row + 8] = acc[h][j][2];
        slot[(tok + 1) * kSlotStride + row + 8] = acc[h][j][3];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_slots_full);
    seg = seg_end;
  }
}

template <int MT>
cudaError_t launch_stream_mt(const CUtensorMap (&maps)[3], const StreamParams& p, int grid, cudaStream_t stream) {
  auto kern = lora_stream_kernel<MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, StreamSmem<MT>::kBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = StreamSmem<MT>::kBytes;
  cfg.stream = stream;
  // programmatic serialisation: the stages start while the rank-r kernel
  // before this one finishes; bf16(s*T) and the counters wait for it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchScope scope(kKindStream, stream);
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], p);
}

}  // namespace

int stream_counter_slots(const LayerDims& d) { return (d.N + kPanelRows - 1) / kPanelRows; }

size_t stream_partial_bytes(int grid) {
  return static_cast<size_t>(2) * grid * kPartialFloats * sizeof(float);
}

// The absmax rows are read by TMA in 16-byte boxes: K a multiple of 256.
bool stream_applies(const LayerDims& d, const Workspace& ws, int sms) {
  if (d.M < 1 || d.M > kStreamMaxTokens || d.K % kStageK != 0) return false;
  if (ws.counters == nullptr || ws.partials == nullptr || ws.counter_cap < stream_counter_slots(d)) return false;
  return ws.partial_bytes >= stream_partial_bytes(sms);
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
  static const bool table_ok = level_table_matches();
  if (!table_ok) return cudaErrorInvalidValue;
  const int mt = d.M <= 8 ? 1 : 2;
  CUtensorMap maps[3];
  // codes [N, K/2] bytes, 128-byte rows of 64-row boxes, swizzled; absmax [N, K/64]
  // fp32, 4 blocks x 64 rows; X [M, K] bf16, 64 features x 8*mt tokens, swizzled
  bool ok = make_tensor_map_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, d.K / 2, d.N, d.K / 2, 128,
                               kPanelRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tensor_map_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, absmax, d.K / 64, d.N, d.K / 16, 4,
                               kPanelRows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
            make_tensor_map_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, d.K, d.M,
                               static_cast<uint64_t>(d.K) * 2, 64, 8 * mt, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  StreamParams p;
  p.B = B;
  p.s_t = ws.s_t;
  p.Y = Y;
  p.partials = ws.partials;
  p.counters = ws.counters;
  p.status = status;
  p.M = d.M;
  p.N = d.N;
  p.r = d.r;
  p.rp = d.rp;
  p.units = d.K / kStageK;
  const int panels = stream_counter_slots(d);
  p.total = static_cast<long long>(panels) * p.units;
  p.whole = panels >= sms ? 1 : 0;
  const int grid = static_cast<int>(p.total < sms ? p.total : sms);
  if (mt == 1) return launch_stream_mt<1>(maps, p, grid, stream);
  return launch_stream_mt<2>(maps, p, grid, stream);
}

}  // namespace qlora
