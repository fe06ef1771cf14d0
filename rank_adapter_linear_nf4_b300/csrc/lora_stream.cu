// lora_stream.cu -- the forward Y = X . W_deq^T + s . (X . A) . B for a handful of
// tokens (M <= 16), where the layer is a stream of its NF4 weight.
//
// Operation: the fused QLoRA linear of the Unsloth pages ("UnSloth加速原理：CUDA内核
// 融合与内存优化", section "内核融合"; "这不是“魔法”是把Unsloth的底层优化逻辑榨干了用",
// section 1), the same result as the main kernel.  With so few tokens the work is
// 0.5625 bytes of codes and absmax per weight element against 2*M flops, so the
// kernel is built around keeping the weight streaming at the HBM rate with as
// few instructions per element as possible:
//
//   * Unit: 16 weight rows (one MMA row group) x a slice of up to 1024 input
//     features (16 NF4 blocks), four items of 256 features.  The CTAs (one per
//     SM, sixteen warps) are shared out evenly among the slices; each takes
//     an equal contiguous range of its slice's items, and each warp an equal
//     contiguous part of its CTA's (at least four items, so a unit has at most
//     two parts).  The X columns of the CTA's slice are copied into shared
//     memory once, at the start.
//   * Each warp streams its own units with its own ring of shared-memory
//     slots and mbarriers: lane 0 issues 2-D TMA copies of 16 rows x 128 bytes
//     of codes (256 input features, 128-byte swizzle) and the matching 16 x 4
//     absmax, four items ahead of the one the warp computes.  No warp waits for
//     another; the weight arrives in long contiguous DRAM reads.
//   * Decode: one shared-memory lookup per code byte in a table of the 256
//     possible bytes -> a pair of bf16 levels, one copy per lane (32 KB, never a
//     bank conflict), straight into the A registers of mma.sync m16n8k16
//     (bf16 -> fp32).  The block's absmax multiplies the block's MMA sum in
//     fp32: the sum of bf16(level[q]) * x * absmax, which is the sum of
//     bf16(level[q] * absmax) * x up to the rounding of the weight (both are
//     within 2^-9 of level[q] * absmax).
//   * The contraction order inside an MMA is free: lane (g, t) of the MMA takes
//     elements 16t .. 16t+15 of a block (its 8 code bytes; k-step s uses bytes
//     2s and 2s+1), and the X fragments are read in that order.
//   * Each part of a unit writes its fp32 partial to its own slot (part 0: the
//     one holding the unit's first item, whose warp also records whether the
//     unit has a second part).  A second kernel, launched right behind with
//     programmatic serialisation, gives each 16-row group to one warp: it adds
//     the group's parts in slice and part order (so the sum does not depend on
//     timing), adds the low-rank term bf16(s*T) . B with mma.sync, and stores
//     the 16 rows of Y.  Its CTA brings its 128 columns of B into shared
//     memory with coalesced loads before it waits for the stream kernel, so
//     that read overlaps the stream's tail.  There are no atomics and no
//     counters.
//   * T comes from the rank-r kernel launched before the stream, which runs
//     beside it; the stream kernel is launched with programmatic serialisation,
//     leaves that kernel's SMs free, and waits for it (griddepcontrol.wait)
//     only at its end, so that the finishing kernel behind it finds T complete.
//
// Every mbarrier wait is bounded (kWaitLimitNs): on expiry the CTA records a
// timeout in the status word and winds down, with no copy left in flight.

#include <cuda_bf16.h>
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "nf4_lut.cuh"
#include "ptx.cuh"

namespace qlora {
namespace {

constexpr int kGroupRows = 16;                // weight rows per unit (one MMA row group)
constexpr int kItemBlocks = 4;                // NF4 blocks per item (one 128-byte code row)
constexpr int kSliceBlocks = 16;              // NF4 blocks per unit (1024 input features)
constexpr int kDepth = 3;                     // items in flight per warp
constexpr int kCodeSlot = kGroupRows * 128;   // bytes of codes per item
constexpr int kAbsSlot = kGroupRows * 16;     // bytes of absmax per item
constexpr uint32_t kLutAlign = 65536;         // the decode table starts on a 64 KB boundary
constexpr int kLutEntry = 256;                // bytes per table entry (32 lane copies in the first 128)
constexpr int kLutBytes = 256 * kLutEntry;
constexpr int kXPitch = kSliceBlocks * 64 * 2 + 16;   // bytes per token row of a staged X slice

// bf16 bit patterns (round to nearest even) of the NF4 levels, in code order:
// the host copy kNF4LevelsHost rounded; launch_stream_fwd checks the two agree.
constexpr uint16_t kLevelBf16[16] = {0xBF80, 0xBF32, 0xBF06, 0xBECA, 0xBE92, 0xBE3D, 0xBDBA, 0x0000,
                                     0x3DA3, 0x3E25, 0x3E7C, 0x3EAD, 0x3EE2, 0x3F10, 0x3F39, 0x3F80};
__constant__ uint16_t c_level_bf16[16] = {0xBF80, 0xBF32, 0xBF06, 0xBECA, 0xBE92, 0xBE3D, 0xBDBA, 0x0000,
                                          0x3DA3, 0x3E25, 0x3E7C, 0x3EAD, 0x3EE2, 0x3F10, 0x3F39, 0x3F80};

// Warps per CTA (one CTA per SM).  (20 warps at one 8-token MMA column block,
// which the registers allow, measured slower than 16.)
template <int MT>
struct StreamCfg {
  static constexpr int kWarps = 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kSlots = kWarps * kDepth;
};

// Shared memory.  The decode table sits on a 64 KB boundary so that one prmt
// forms a lookup address (table | byte << 8 | lane << 2); the code slots
// (1024-aligned, for the 128-byte swizzle) fill the space below it and, with
// the absmax slots, the staged X slice and the barriers, the space above.
template <int MT>
struct StreamLayout {
  static constexpr int kSlots = StreamCfg<MT>::kSlots;
  static constexpr int kXRows = 8 * MT;   // token rows of the X slice
  uint32_t code_lo, n_lo;   // slots 0 .. n_lo-1 below the table
  uint32_t lut;
  uint32_t code_hi;         // slots n_lo .. kSlots-1 above it
  uint32_t abs, x, bar, end;
  __device__ __forceinline__ explicit StreamLayout(uint32_t window) {
    code_lo = (window + 1023u) & ~1023u;
    lut = (code_lo + kLutAlign - 1u) & ~(kLutAlign - 1u);
    uint32_t n = (lut - code_lo) / kCodeSlot;
    n -= n % kDepth;                                   // a warp's ring never straddles the table
    n_lo = n < static_cast<uint32_t>(kSlots) ? n : static_cast<uint32_t>(kSlots);
    code_hi = lut + kLutBytes;
    abs = code_hi + (kSlots - n_lo) * kCodeSlot;
    x = abs + kSlots * kAbsSlot;
    bar = x + kXRows * kXPitch;
    end = bar + 8u * (kSlots + 1);
  }
  __device__ __forceinline__ uint32_t ring(int warp) const {
    const uint32_t j = static_cast<uint32_t>(warp * kDepth);
    return j < n_lo ? code_lo + j * kCodeSlot : code_hi + (j - n_lo) * kCodeSlot;
  }
};
static_assert(kCodeSlot % 1024 == 0 && kLutBytes % 1024 == 0, "code slots keep the 128-byte swizzle alignment");
static_assert(kXPitch % 16 == 0 && kAbsSlot % 16 == 0, "bulk copies need 16-byte alignment");

struct StreamParams {
  const uint16_t* X;        // [M, K] bf16
  const uint16_t* B;        // [r, N] bf16
  const uint16_t* s_t;      // [M, rp] bf16(s*T), zero columns r..rp-1
  uint16_t* Y;              // [M, N] bf16
  float* partials;          // two slots (parts) of 128 * MT floats per unit
  int* unit_parts;          // [units]: 1 or 2, written each call by the warp holding part 0
  int* status;
  int M, K, N, r, rp;
  int kb;                   // NF4 blocks per row: K / 64
  int groups;               // 16-row groups: ceil(N / 16)
  int slices;               // ceil(kb / 16)
  int units;                // slices * groups
  int cps;                  // CTAs per slice
};

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
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

// The pair-table word of code byte i of w from this lane's copy: the address
// is the table base with the byte in bits 8-15 and 4 * lane in bits 0-7
// (lut_lane), assembled by one prmt with selector 0x7604 | i << 4.
__device__ __forceinline__ uint32_t lut_pair(uint32_t lut_lane, uint32_t w, uint32_t sel) {
  return lds32(prmt(w, lut_lane, sel));
}

// Blocks of slice s.
__device__ __forceinline__ int slice_blocks(const StreamParams& p, int s) {
  return min(kSliceBlocks, p.kb - s * kSliceBlocks);
}

// The static split of slice s's items: CTA `sub` of the slice takes items
// [n*sub/cps, n*(sub+1)/cps), and its `active` warps equal parts of those.
struct SliceSplit {
  int n;        // items of the slice
  __device__ __forceinline__ int cta_begin(const StreamParams& p, int sub) const {
    return static_cast<int>(static_cast<int64_t>(n) * sub / p.cps);
  }
  template <int W>
  __device__ __forceinline__ static int active_warps(int n_cta) { return min(W, max(1, n_cta / kItemBlocks)); }
};

// One item's MMAs: acc += absmax * (codes of 16 rows x 4 blocks) . X.  Token
// rows at or past M are not read: their lanes' X fragments stay zero (and
// their MMA columns are never stored).
template <int MT>
__device__ __forceinline__ void compute_item(uint32_t code_slot, uint32_t abs_slot, const uint8_t* x_row0, int blk0,
                                             uint32_t lut_lane, int g4, int t, const bool (&live)[MT],
                                             uint4 (&x)[MT][2], float (&acc)[MT][4]) {
  const uint32_t ra = static_cast<uint32_t>(g4), rb = static_cast<uint32_t>(g4 + 8);
  const uint4 am_a4 = ld_shared_v4(abs_slot + ra * 16u);   // the item's four block scales, rows g and g+8
  const uint4 am_b4 = ld_shared_v4(abs_slot + rb * 16u);
#pragma unroll
  for (int blk = 0; blk < kItemBlocks; ++blk) {
    // rows g and g+8, bytes 8t .. 8t+7 of block blk: 16-byte chunk 2*blk + t/2,
    // swizzled by the row (128-byte swizzle; rows g and g+8 swizzle alike), half t%2 of it
    const uint32_t chunk = static_cast<uint32_t>(2 * blk + (t >> 1));
    const uint32_t ca_addr = code_slot + ra * 128u + ((chunk ^ (ra & 7u)) << 4) + 8u * (t & 1);
    const uint2 ca = lds64(ca_addr);
    const uint2 cb = lds64(ca_addr + 1024u);
    const float am_a = __uint_as_float(blk == 0 ? am_a4.x : blk == 1 ? am_a4.y : blk == 2 ? am_a4.z : am_a4.w);
    const float am_b = __uint_as_float(blk == 0 ? am_b4.x : blk == 1 ? am_b4.y : blk == 2 ? am_b4.z : am_b4.w);
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      // a lane of an absent token keeps the zeros its fragment started with
      const uint4* src = reinterpret_cast<const uint4*>(x_row0 + j * 8 * kXPitch + ((blk0 + blk) * 64 + 16 * t) * 2);
      if (live[j]) {
        x[j][0] = src[0];
        x[j][1] = src[1];
      }
    }
    float d[MT][4];
#pragma unroll
    for (int j = 0; j < MT; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.0f;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      // k-step s: code bytes 2s (fragment columns 2t, 2t+1) and 2s+1 (2t+8, 2t+9)
      const uint32_t wa = s < 2 ? ca.x : ca.y, wb = s < 2 ? cb.x : cb.y;
      const uint32_t sel0 = 0x7604u | (static_cast<uint32_t>((2 * s) & 3) << 4);
      const uint32_t sel1 = 0x7604u | (static_cast<uint32_t>((2 * s + 1) & 3) << 4);
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
      acc[j][0] = fmaf(am_a, d[j][0], acc[j][0]);
      acc[j][1] = fmaf(am_a, d[j][1], acc[j][1]);
      acc[j][2] = fmaf(am_b, d[j][2], acc[j][2]);
      acc[j][3] = fmaf(am_b, d[j][3], acc[j][3]);
    }
  }
}

template <int MT>
__device__ __forceinline__ float* slot_ptr(const StreamParams& p, int unit, int part, int lane) {
  return p.partials + (static_cast<int64_t>(unit) * 2 + part) * (128 * MT) + lane * 4;
}

constexpr int kFinWarps = 8;                      // 16-row groups per finishing CTA
constexpr int kFinCols = kFinWarps * kGroupRows;   // columns of B per finishing CTA
constexpr int kFinBPitch = kFinCols * 2 + 16;      // bytes per rank row of the staged B tile

// Finishes row group `group` (warp `gw` of its CTA): its units' sums in slice
// and part order, the low-rank term with B from the CTA's tile (b_tile: rp rows
// of kFinCols columns) and bf16(s*T) from s_t (16 rows of rp), then Y.
template <int MT, int RP>
__device__ __forceinline__ void finish_group(const StreamParams& p, int group, int gw, int lane, uint32_t b_tile,
                                             uint32_t s_t) {
  const int g4 = lane >> 2, t = lane & 3;
  const int na = group * kGroupRows + g4, nb = na + 8;
  float acc[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
  // both parts' slots are read together with the part count; a second part
  // that was not written this call is ignored (never added)
#pragma unroll 4
  for (int s = 0; s < p.slices; ++s) {
    const int uid = s * p.groups + group;
    const int parts = __ldcg(p.unit_parts + uid);
    const float* src0 = slot_ptr<MT>(p, uid, 0, lane);
    const float* src1 = slot_ptr<MT>(p, uid, 1, lane);
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src0 + j * 128));
      const float4 w = __ldcg(reinterpret_cast<const float4*>(src1 + j * 128));
      const bool two = parts == 2;
      acc[j][0] += two ? v.x + w.x : v.x;
      acc[j][1] += two ? v.y + w.y : v.y;
      acc[j][2] += two ? v.z + w.z : v.z;
      acc[j][3] += two ? v.w + w.w : v.w;
    }
  }
  // low-rank term: D += B^T (rows n, columns j) . bf16(s*T)^T (rows j, columns tokens)
  const uint32_t col = static_cast<uint32_t>(gw * kGroupRows + g4) * 2u;   // column g of the group in the tile
#pragma unroll
  for (int ks = 0; ks < RP / 16; ++ks) {
    const uint32_t r0 = b_tile + static_cast<uint32_t>(16 * ks + 2 * t) * kFinBPitch + col;
    auto u16 = [](uint32_t addr) -> uint32_t {
      uint16_t v;
      asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
      return v;
    };
    const uint32_t a[4] = {u16(r0) | (u16(r0 + kFinBPitch) << 16), u16(r0 + 16) | (u16(r0 + kFinBPitch + 16) << 16),
                           u16(r0 + 8 * kFinBPitch) | (u16(r0 + 9 * kFinBPitch) << 16),
                           u16(r0 + 8 * kFinBPitch + 16) | (u16(r0 + 9 * kFinBPitch + 16) << 16)};
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      const uint32_t trow = s_t + static_cast<uint32_t>((8 * j + g4) * (RP * 2 + 16) + (16 * ks + 2 * t) * 2);
      mma_16816(acc[j], a, lds32(trow), lds32(trow + 16));
    }
  }
  // Y: c0, c1 -> row g, tokens 2t, 2t+1 of the half; c2, c3 -> row g+8
#pragma unroll
  for (int j = 0; j < MT; ++j) {
    const int tok = 8 * j + 2 * t;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = (e < 2) ? na : nb, tk = tok + (e & 1);
      if (n < p.N && tk < p.M)
        p.Y[static_cast<int64_t>(tk) * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j][e]));
    }
  }
}

template <int MT>
__global__ void __launch_bounds__(StreamCfg<MT>::kThreads, 1)
    lora_stream_kernel(const __grid_constant__ CUtensorMap map_codes,   // [N, K/2] bytes, box {128, 16}, 128-B swizzle
                       const __grid_constant__ CUtensorMap map_abs,     // [N, K/64] fp32, box {4, 16}
                       const StreamParams p) {
  using L = StreamLayout<MT>;
  constexpr int kWarps = StreamCfg<MT>::kWarps;
  constexpr int kThreads = StreamCfg<MT>::kThreads;
  constexpr int kSlots = StreamCfg<MT>::kSlots;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  const uint32_t window = smem_u32(smem_raw);
  const L lay(window);
  uint32_t dyn_bytes;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
  if (lay.end > window + dyn_bytes) {
    // the layout needs more shared memory than the launch gave: compute nothing
    if (threadIdx.x == 0) atomicExch(p.status, kStatusInternal);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g4 = lane >> 2, t = lane & 3;

  // this CTA's slice and items, and this warp's part of them; every unit of
  // the slice has the same number of items (ipu), so the cursors below step
  // through (group, item) pairs without divisions
  const int slice = blockIdx.x / p.cps, sub = blockIdx.x % p.cps;
  const int ipu = slice_blocks(p, slice) / kItemBlocks;
  const SliceSplit split{p.groups * ipu};
  const int i_begin = split.cta_begin(p, sub), i_end = split.cta_begin(p, sub + 1);
  const int n_cta = i_end - i_begin;
  const int active = SliceSplit::active_warps<kWarps>(n_cta);   // at least four items per warp
  const int w_lo = warp < active ? i_begin + n_cta * warp / active : i_end;
  const int w_hi = warp < active ? i_begin + n_cta * (warp + 1) / active : i_end;
  const int n_items = w_hi - w_lo;
  const uint32_t x_bar = lay.bar + 8u * kSlots;
  auto full = [&](int slot) { return lay.bar + 8u * static_cast<uint32_t>(warp * kDepth + slot); };
  Abort ab{&s_abort, p.status};

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kSlots; ++i) mbar_init(lay.bar + 8u * i, 1);
    mbar_init(x_bar, 1);
    fence_barrier_init();
  }
  // the decode table: entry v, lane l holds bf16(level[v >> 4]) (the byte's
  // first element) in its low half and bf16(level[v & 15]) in its high half;
  // four lane copies per 16-byte store
  for (int i = threadIdx.x; i < 256 * 8; i += kThreads) {
    const int v = i >> 3;
    const uint32_t w =
        static_cast<uint32_t>(c_level_bf16[v >> 4]) | (static_cast<uint32_t>(c_level_bf16[v & 15]) << 16);
    st_shared_v4(lay.lut + static_cast<uint32_t>(v * kLutEntry + (i & 7) * 16), make_uint4(w, w, w, w));
  }
  __syncthreads();

  if (threadIdx.x == 0) {
    // X columns of the CTA's slice, one bulk copy per token row
    const uint32_t row_bytes = static_cast<uint32_t>(slice_blocks(p, slice) * 128);
    mbar_arrive_expect_tx(x_bar, row_bytes * static_cast<uint32_t>(p.M));
    for (int tok = 0; tok < p.M; ++tok)
      bulk_load_1d(lay.x + static_cast<uint32_t>(tok * kXPitch),
                   p.X + static_cast<int64_t>(tok) * p.K + slice * (kSliceBlocks * 64), row_bytes, x_bar);
  }

  const uint32_t code_ring = lay.ring(warp);
  const uint32_t abs_ring = lay.abs + static_cast<uint32_t>(warp * kDepth * kAbsSlot);
  auto issue = [&](int g, int it, int slot) {
    const int blk0 = slice * kSliceBlocks + it * kItemBlocks;
    mbar_arrive_expect_tx(full(slot), kCodeSlot + kAbsSlot);
    tma_load_2d(code_ring + slot * kCodeSlot, &map_codes, full(slot), blk0 * 32, g * kGroupRows);
    tma_load_2d(abs_ring + slot * kAbsSlot, &map_abs, full(slot), blk0, g * kGroupRows);
  };
  auto step = [&](int& g, int& it) {
    if (++it == ipu) {
      it = 0;
      ++g;
    }
  };

  // (group, item) of the item computed and, on lane 0, of the next one to load
  int cg = w_lo / ipu, cit = w_lo % ipu;
  int lg = cg, lit = cit;
  if (lane == 0) {
    tma_prefetch_map(&map_codes);
    tma_prefetch_map(&map_abs);
    for (int q = 0; q < kDepth && q < n_items; ++q) {
      issue(lg, lit, q);
      step(lg, lit);
    }
  }
  // every lane acquires the bulk-copied X itself
  bool ok = mbar_wait(x_bar, 0, ab);
  const uint32_t lut_lane = lay.lut | (static_cast<uint32_t>(lane) << 2);
  const uint8_t* const x_row0 = smem_raw + (lay.x - window) + g4 * kXPitch;
  bool live[MT];
  uint4 xfrag[MT][2];
#pragma unroll
  for (int j = 0; j < MT; ++j) {
    live[j] = 8 * j + g4 < p.M;
    xfrag[j][0] = xfrag[j][1] = make_uint4(0u, 0u, 0u, 0u);
  }
  float acc[MT][4];
#pragma unroll
  for (int j = 0; j < MT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
  int seg_part = cit == 0 ? 0 : 1;   // the current part of a unit
  int k = 0;
  int slot = 0;
  uint32_t phase = 0;
  for (; ok && k < n_items; ++k) {
    if (!__all_sync(0xffffffffu, mbar_wait(full(slot), phase, ab))) {
      ok = false;
      break;
    }
    compute_item<MT>(code_ring + slot * kCodeSlot, abs_ring + slot * kAbsSlot, x_row0, cit * kItemBlocks, lut_lane,
                     g4, t, live, xfrag, acc);
    // the slot's codes have been read by every lane: refill it kDepth items ahead
    __syncwarp();
    if (lane == 0 && k + kDepth < n_items) {
      fence_proxy_async_smem();
      issue(lg, lit, slot);
      step(lg, lit);
    }
    if (cit + 1 == ipu || k + 1 == n_items) {
      // the end of this warp's part of the unit (part 0 records whether it is the whole unit)
      const int u = slice * p.groups + cg;
      if (seg_part == 0 && lane == 0) p.unit_parts[u] = cit + 1 == ipu ? 1 : 2;
      float* dst = slot_ptr<MT>(p, u, seg_part, lane);
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        __stcg(reinterpret_cast<float4*>(dst + j * 128), make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]));
        acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
      }
      seg_part = 0;
    }
    step(cg, cit);
    if (++slot == kDepth) {
      slot = 0;
      phase ^= 1u;
    }
  }
  if (!ok) {
    // a wait ran out: let the copies this CTA issued land before it exits
    if (lane == 0)
      for (int q = k; q < n_items && q < k + kDepth; ++q) mbar_wait(full(q % kDepth), (q / kDepth) & 1, ab, false);
    if (threadIdx.x == 0) mbar_wait(x_bar, 0, ab, false);
    return;
  }

  // the finishing kernel behind this one reads T: this grid completes only
  // after the rank-r kernel before it has; then let the finishing kernel start
  griddep_wait();
  griddep_launch_dependents();
}

// The 16-row groups, one per warp: parts in slice order, the low-rank term, Y.
template <int MT, int RP>
__global__ void __launch_bounds__(kFinWarps * 32) lora_stream_finish_kernel(const StreamParams p) {
  __shared__ __align__(16) uint8_t b_tile[RP * kFinBPitch];          // B [rp][this CTA's 128 columns]
  __shared__ __align__(16) uint8_t t_tile[16 * (RP * 2 + 16)];       // bf16(s*T) [16 tokens][rp]
  const int n0 = static_cast<int>(blockIdx.x) * kFinCols;
  // the next call's first kernel may be scheduled now: it waits for this grid
  // before it touches global memory
  if (threadIdx.x == 0) griddep_launch_dependents();
  // B is an input of the call: bring this CTA's columns in while the stream kernel finishes
  for (int i = threadIdx.x; i < RP * (kFinCols / 8); i += kFinWarps * 32) {
    const int j = i / (kFinCols / 8), c = (i % (kFinCols / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < p.r && n0 + c < p.N) v = ldg_nc_v4(p.B + static_cast<int64_t>(j) * p.N + n0 + c);
    st_shared_v4(smem_u32(b_tile) + static_cast<uint32_t>(j * kFinBPitch + c * 2), v);
  }
  // the stream kernel before this one wrote the partials (and completed after the rank-r kernel)
  griddep_wait();
  for (int i = threadIdx.x; i < 16 * (RP / 8); i += kFinWarps * 32) {
    const int tok = i / (RP / 8), c = (i % (RP / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (tok < p.M) v = *reinterpret_cast<const uint4*>(p.s_t + static_cast<int64_t>(tok) * p.rp + c);
    st_shared_v4(smem_u32(t_tile) + static_cast<uint32_t>(tok * (RP * 2 + 16) + c * 2), v);
  }
  __syncthreads();
  const int gw = static_cast<int>(threadIdx.x >> 5);
  const int g = static_cast<int>(blockIdx.x) * kFinWarps + gw;
  if (g < p.groups) finish_group<MT, RP>(p, g, gw, threadIdx.x & 31, smem_u32(b_tile), smem_u32(t_tile));
}

// The opt-in shared memory per block less the kernel's static shared memory.
int stream_dynamic_smem(const void* kern) {
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return -1;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return -1;
  return optin - static_cast<int>(fa.sharedSizeBytes);
}

template <int MT>
cudaError_t launch_stream_mt(const CUtensorMap (&maps)[2], const StreamParams& p, int grid, cudaStream_t stream) {
  auto kern = lora_stream_kernel<MT>;
  // all the shared memory a CTA may have: the layout is placed around a 64 KB
  // boundary of the CTA's window, which the kernel checks it has room for
  static const int dyn_bytes = stream_dynamic_smem(reinterpret_cast<const void*>(kern));
  if (dyn_bytes <= 0) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(StreamCfg<MT>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn_bytes;
  cfg.stream = stream;
  // programmatic serialisation: the weight stream starts while the rank-r
  // kernel before this one finishes; bf16(s*T) and the counters wait for it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    LaunchScope scope(kKindStream, stream);
    e = cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], p);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t fin = cfg;
  fin.gridDim = dim3((p.groups + kFinWarps - 1) / kFinWarps, 1, 1);
  fin.blockDim = dim3(kFinWarps * 32, 1, 1);
  fin.dynamicSmemBytes = 0;
  LaunchScope scope(kKindStreamFinish, stream);
  if (p.rp == 64) return cudaLaunchKernelEx(&fin, lora_stream_finish_kernel<MT, 64>, p);
  return cudaLaunchKernelEx(&fin, lora_stream_finish_kernel<MT, 128>, p);
}

int stream_groups(const LayerDims& d) { return (d.N + kGroupRows - 1) / kGroupRows; }

int stream_units(const LayerDims& d) {
  const int kb = d.K / 64;
  return ((kb + kSliceBlocks - 1) / kSliceBlocks) * stream_groups(d);
}

}  // namespace

int stream_counter_slots(const LayerDims& d) {
  (void)d;
  return 0;   // the token-stream forward uses no counters
}

namespace {
size_t stream_slot_bytes(const LayerDims& d) {
  const int mt = d.M <= 8 ? 1 : 2;
  // two slots per unit, then a part count per unit
  return (static_cast<size_t>(stream_units(d)) * (2 * 128 * mt * sizeof(float) + sizeof(int)) + 15) & ~size_t(15);
}
}  // namespace

size_t stream_partial_bytes(const LayerDims& d, int sms) {
  (void)sms;
  return stream_slot_bytes(d);
}

// The absmax rows are read by TMA in 16-byte boxes, and an item is four blocks:
// K a multiple of 256; and there must be a CTA for every slice.
bool stream_applies(const LayerDims& d, const Workspace& ws, int sms) {
  if (d.M < 1 || d.M > kStreamMaxTokens || d.K % 256 != 0 || d.rp > 128) return false;
  if ((d.K / 64 + kSliceBlocks - 1) / kSliceBlocks > sms - kStreamReservedSms) return false;
  if (ws.partials == nullptr) return false;
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
  static const bool table_ok = level_table_matches();
  if (!table_ok) return cudaErrorInvalidValue;
  CUtensorMap maps[2];
  // codes [N, K/2] bytes: 128-byte rows of 16-row boxes, swizzled; absmax [N, K/64] fp32, 4 blocks x 16 rows
  bool ok = make_tensor_map_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, d.K / 2, d.N, d.K / 2, 128,
                               kGroupRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_tensor_map_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, absmax, d.K / 64, d.N, d.K / 16, 4,
                               kGroupRows, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  StreamParams p;
  p.X = X;
  p.B = B;
  p.s_t = ws.s_t;
  p.Y = Y;
  p.partials = ws.partials;
  p.unit_parts = reinterpret_cast<int*>(ws.partials + static_cast<size_t>(stream_units(d)) * 2 * 128 * (d.M <= 8 ? 1 : 2));
  p.status = status;
  p.M = d.M;
  p.K = d.K;
  p.N = d.N;
  p.r = d.r;
  p.rp = d.rp;
  p.kb = d.K / 64;
  p.groups = stream_groups(d);
  p.slices = (p.kb + kSliceBlocks - 1) / kSliceBlocks;
  p.units = p.slices * p.groups;
  // the CTAs are shared out among the slices (at least four items each), and
  // leave the rank-r kernel's SMs free so that every CTA starts at once beside it
  const int slice_items = p.groups * (kSliceBlocks / kItemBlocks);
  p.cps = std::max(1, std::min((sms - kStreamReservedSms) / p.slices, slice_items / kItemBlocks));
  const int grid = p.slices * p.cps;
  if (d.M <= 8) return launch_stream_mt<1>(maps, p, grid, stream);
  return launch_stream_mt<2>(maps, p, grid, stream);
}

}  // namespace qlora
