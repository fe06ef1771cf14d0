// lora_merge.cu -- the merged 16-bit weight W_merged = bf16(W_deq + s . (A . B)^T).
//
// (Unsloth pages: "这不是“魔法”是把Unsloth的底层优化逻辑榨干了用", section 4:
// save_pretrained_merged(..., "merged_16bit"), the adapter folded into the base
// weight for export.  Re-quantising the merged weight to NF4 is
// qlora_quantize_nf4 on this kernel's output.)
//
// One CTA per 128 x 128 tile of W_merged [d_out, d_in] (rows n, columns k):
//   * the rank-r product of the tile is one tcgen05 MMA chain in TMEM,
//       D[128 n x 128 k] = B^T tile [128 n x rp] . A^T tile [rp x 128 k],
//     with B^T as the MN-major A operand (rows of B [r, d_out] run along n) and
//     A^T as the K-major B operand (rows of A [d_in, r] run along the rank);
//     the threads stage both into 128-byte-swizzled shared memory, zero past r
//     and past the matrix edges, so any rank 1..128 and any alignment of A work;
//   * the epilogue adds the tile's NF4 expansion -- the per-block table of
//     qlora_dequant_nf4, so W_deq is that kernel's output bit for bit -- rounds
//     once to bf16, out = bf16_rn(fma(s, D, W_deq)), stages the tile in the
//     operands' shared memory (128-byte swizzle) and writes it with TMA stores.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "nf4_lut.cuh"
#include "ptx.cuh"

namespace qlora {

namespace {

constexpr int kMergeTile = 128;     // tile rows (n) and columns (k)
constexpr int kMergeThreads = 128;  // thread t: staging row t, TMEM lane / output row t

struct MergeParams {
  const uint8_t* packed;   // [N, K/2]
  const float* absmax;     // [N, K/64]
  const uint16_t* A;       // [K, r] bf16
  const uint16_t* B;       // [r, N] bf16
  int N, K, r;
  float s;
  int a_vec;               // A 16-byte aligned with r % 8 == 0: 16-byte loads
  int b_vec;               // B 16-byte aligned: 16-byte loads (N % 8 == 0 always)
  int* status;
};

template <int RP>
struct MergeSmem {
  static constexpr int kChunks = RP / 64;           // 64-wide chunks of the rank
  static constexpr int kChunkBytes = 128 * 128;     // 128 rows (or 2 x 64 columns) x 64 bf16
  static constexpr int kBtOffset = 0;               // B^T operand, MN-major
  static constexpr int kAtOffset = kChunks * kChunkBytes;   // A^T operand, K-major
  static constexpr int kStageOffset = 0;            // output tile staging, reuses the operands
  static constexpr int kBarOffset = 2 * kChunks * kChunkBytes;
  // at least 46 KB: at most 4 CTAs per SM (5 x 47 KB exceeds the 228 KB), so their
  // 128-column TMEM allocations always fit in the 512 columns
  static constexpr int kBytes = (kBarOffset + 64 + 1024) > 46 * 1024 ? (kBarOffset + 64 + 1024) : 46 * 1024;
  static_assert(kBarOffset >= 2 * kChunkBytes, "the output staging fits in the operand space");
};

__device__ __forceinline__ uint16_t ld_bf16(const uint16_t* p) {
  return __ldg(reinterpret_cast<const unsigned short*>(p));
}

// Eight consecutive bf16 of a row, zero outside [0, limit): one 16-byte load when
// `vec` (aligned), else element by element.
__device__ __forceinline__ uint4 ld_bf16x8(const uint16_t* row, int first, int limit, bool vec) {
  if (vec && first + 8 <= limit) return ldg_nc_v4(reinterpret_cast<const uint4*>(row + first));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (first + e < limit) w[e >> 1] |= static_cast<uint32_t>(ld_bf16(row + first + e)) << (16 * (e & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int RP>
__global__ void __launch_bounds__(kMergeThreads) lora_merge_kernel(const __grid_constant__ CUtensorMap map_out,
                                                                 const MergeParams p) {
  using S = MergeSmem<RP>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar = base + S::kBarOffset;
  const int t = threadIdx.x, warp = t >> 5;
  const int k0 = blockIdx.x * kMergeTile, n0 = blockIdx.y * kMergeTile;
  Abort ab{&s_abort, p.status};

  if (t == 0) {
    s_abort = 0;
    mbar_init(bar, 1);
    fence_barrier_init();
    tma_prefetch_map(&map_out);
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), kMergeTile);

  // this thread's output row n = n0 + t: its 128 codes (64 B) and two absmax values,
  // requested now so that their latency hides behind the operand staging and the MMAs
  const int n = n0 + t;
  const int kblocks = p.K >> 6;
  uint4 codes[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                    make_uint4(0u, 0u, 0u, 0u)};
  float amax[2] = {0.f, 0.f};
  if (n < p.N) {
    const uint4* crow = reinterpret_cast<const uint4*>(p.packed + static_cast<int64_t>(n) * (p.K / 2) + k0 / 2);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (k0 + 64 * h < p.K) {
        codes[2 * h] = ldg_nc_v4(crow + 2 * h);
        codes[2 * h + 1] = ldg_nc_v4(crow + 2 * h + 1);
        amax[h] = ldg_nc_f32(p.absmax + static_cast<int64_t>(n) * kblocks + (k0 >> 6) + h);
      }
    }
  }

  // ---- stage B^T (MN-major): rank row j, columns n0..n0+127 as two 64-column blocks
  //      of 128 B; 16-B chunk q of row j sits at (q % 8) ^ (j & 7).  Consecutive threads
  //      take consecutive 16-B chunks of a row: the loads are coalesced.
  for (int e = t; e < RP * 16; e += kMergeThreads) {
    const int j = e >> 4, q = e & 15;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < p.r) v = ld_bf16x8(p.B + static_cast<int64_t>(j) * p.N, n0 + 8 * q, p.N, p.b_vec != 0);
    const uint32_t row = base + S::kBtOffset + (j >> 6) * S::kChunkBytes + (j & 63) * 128;
    st_shared_v4(row + static_cast<uint32_t>(q >> 3) * 8192u + (((q & 7) ^ (j & 7)) << 4), v);
  }
  // ---- stage A^T (K-major): column k = k0 + kl, rank chunk c, 16-B chunk q at q ^ (kl & 7).
  //      The tile's rows of A are one contiguous block: consecutive threads, consecutive chunks.
  for (int e = t; e < kMergeTile * (RP / 8); e += kMergeThreads) {
    const int kl = e / (RP / 8), q = e % (RP / 8);
    const int k = k0 + kl;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (k < p.K) v = ld_bf16x8(p.A + static_cast<int64_t>(k) * p.r, 8 * q, p.r, p.a_vec != 0);
    const uint32_t row = base + S::kAtOffset + (q >> 3) * S::kChunkBytes + kl * 128;
    st_shared_v4(row + (((q & 7) ^ (kl & 7)) << 4), v);
  }
  fence_proxy_async_smem();   // the tensor core reads what the threads wrote
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (t == 0) {
    constexpr uint32_t idesc = umma_idesc_bf16(kMergeTile, kMergeTile, 1, 0);
#pragma unroll
    for (int c = 0; c < S::kChunks; ++c) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = sw128_desc(base + S::kBtOffset + c * S::kChunkBytes + kk * 2048, 8192, 1024);
        const uint64_t bd = sw128_desc(base + S::kAtOffset + c * S::kChunkBytes + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (c | kk) != 0 ? 1u : 0u);
      }
    }
    umma_commit(bar);
  }
  __syncwarp();
  // the MMAs have read the operands once this completes: their space becomes the staging
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, 0, ab, false));
  tc_fence_after_sync();

  // ---- epilogue: row n = n0 + t, 32 columns at a time, into the 128-B-swizzled staging
  //      (two [128 rows][64 columns] halves), then two TMA stores
  Nf4BlockTable tab;
#pragma unroll
  for (int cc = 0; cc < kMergeTile / 32; ++cc) {
    uint32_t v[32];
    tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + 32 * cc, v);
    tmem_ld_wait();
    const int k = k0 + 32 * cc;
    if (!ok || n >= p.N || k >= p.K) continue;   // outside the matrix: the TMA store clips it
    if ((cc & 1) == 0) tab = nf4_block_table(amax[cc >> 1]);
    const uint4 c16 = codes[cc];
    const uint32_t words[4] = {c16.x, c16.y, c16.z, c16.w};
    const uint32_t half = base + S::kStageOffset + static_cast<uint32_t>(cc >> 1) * S::kChunkBytes + t * 128;
#pragma unroll
    for (int wq = 0; wq < 4; ++wq) {
      const uint4 wd = nf4_expand8(words[wq], tab);   // bf16 pairs, elements 8wq..8wq+7
      const uint32_t pr[4] = {wd.x, wd.y, wd.z, wd.w};
      uint32_t o[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float w0 = __uint_as_float(pr[h] << 16), w1 = __uint_as_float(pr[h] & 0xFFFF0000u);
        const float a0 = __uint_as_float(v[8 * wq + 2 * h]), a1 = __uint_as_float(v[8 * wq + 2 * h + 1]);
        o[h] = pack_bf16x2(fmaf(p.s, a0, w0), fmaf(p.s, a1, w1));
      }
      const uint32_t chunk = static_cast<uint32_t>((cc & 1) * 4 + wq);   // 16-B chunk within the 128-B row
      st_shared_v4(half + ((chunk ^ (t & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  if (t == 0 && ok) {
    tma_store_2d(&map_out, base + S::kStageOffset, k0, n0);
    if (k0 + 64 < p.K) tma_store_2d(&map_out, base + S::kStageOffset + S::kChunkBytes, k0 + 64, n0);
    tma_store_commit();
    tma_store_wait_read_all();   // the staging must outlive the reads, not the writes
  }
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kMergeTile);
  }
}

// ---------------------------------------------------------------------------
// Persistent form (r % 8 == 0, A and B 16-byte aligned): one CTA per SM takes
// a contiguous run of 128 x 128 output tiles in row-block order, so its B^T
// operand is loaded once per row block.  Warp 16 (one lane) loads A^T tiles by
// TMA into a two-slot ring and issues each tile's rank-r MMA into one of two
// TMEM accumulators; warps 0-15 are the epilogue (TMEM lane = tile row; warps
// w, w + 4, w + 8, w + 12 take 32 columns each): while tile i's MMA runs they
// finish tile i - 1 -- its codes and absmax were loaded from global memory two
// tiles ahead -- into one of two staging buffers, which a TMA store writes out
// while the next tile is computed.
constexpr int kMpEpiWarps = 16;
constexpr int kMpThreads = (kMpEpiWarps + 1) * 32;
constexpr int kMpASlots = 2;

template <int RP>
struct MergePSmem {
  static constexpr int kChunks = RP / 64;
  static constexpr int kOpBytes = kChunks * 16384;            // one operand (B^T or an A^T tile)
  static constexpr int kBtOff = 0;
  static constexpr int kAOff = kBtOff + kOpBytes;
  static constexpr int kStageOff = kAOff + kMpASlots * kOpBytes;   // 16 warps x two 4 KB output stagings
  static constexpr int kBarOff = kStageOff + kMpEpiWarps * 8192;
  // bars: a_full[2], a_empty[2], tmem_full[2], tmem_empty[2], bt_full, bt_free, drain
  static constexpr int kBytes = kBarOff + 8 * 11 + 1024;
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kStageOff % 1024 == 0, "stagings keep the 128-byte swizzle alignment");
};

template <int RP>
__global__ void __launch_bounds__(kMpThreads, 1)
    lora_merge_persistent_kernel(const __grid_constant__ CUtensorMap map_out,   // W_out [N, K] bf16, box {64, 32}, 128-B swizzle
                                 const __grid_constant__ CUtensorMap map_a,     // A [K, r] bf16, box {64, 128}, SW128
                                 const __grid_constant__ CUtensorMap map_b,     // B [r, N] bf16, box {64, 64}, SW128
                                 const MergeParams p, int k_tiles, int tiles) {
  using S = MergePSmem<RP>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t bars = base + S::kBarOff;
  auto a_full = [&](int s) { return bars + 8u * s; };
  auto a_empty = [&](int s) { return bars + 16u + 8u * s; };
  auto tmem_full = [&](int b) { return bars + 32u + 8u * b; };
  auto tmem_empty = [&](int b) { return bars + 48u + 8u * b; };
  const uint32_t bt_full = bars + 64u, bt_free = bars + 72u, drain = bars + 80u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Abort ab{&s_abort, p.status};
  // this CTA's tiles: [t_begin, t_end) of the row-block-major order
  const int t_begin = static_cast<int>(static_cast<int64_t>(tiles) * blockIdx.x / gridDim.x);
  const int t_end = static_cast<int>(static_cast<int64_t>(tiles) * (blockIdx.x + 1) / gridDim.x);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kMpASlots; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(a_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tmem_full(b), 1);
      mbar_init(tmem_empty(b), kMpEpiWarps / 2);   // the half of the epilogue warps that finishes it
    }
    mbar_init(bt_full, 1);
    mbar_init(bt_free, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), 256);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == kMpEpiWarps) {
    // ---------------- A^T / B^T loads and the MMAs (one lane)
    if (lane == 0) {
      tma_prefetch_map(&map_a);
      tma_prefetch_map(&map_b);
      tma_prefetch_map(&map_out);
      auto load_a = [&](int tile, int slot) {
        const int k0 = (tile % k_tiles) * kMergeTile;
        mbar_arrive_expect_tx(a_full(slot), S::kOpBytes);
#pragma unroll
        for (int c = 0; c < S::kChunks; ++c)
          tma_load_2d(base + S::kAOff + slot * S::kOpBytes + c * 16384, &map_a, a_full(slot), c * 64, k0);
      };
      auto load_bt = [&](int nb) {
        const int n0 = nb * kMergeTile;
        mbar_arrive_expect_tx(bt_full, S::kOpBytes);
#pragma unroll
        for (int c = 0; c < S::kChunks; ++c)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(base + S::kBtOff + c * 16384 + h * 8192, &map_b, bt_full, n0 + 64 * h, c * 64);
      };
      int loaded = 0;   // A tiles requested (relative to t_begin)
      for (; loaded < kMpASlots && t_begin + loaded < t_end; ++loaded) load_a(t_begin + loaded, loaded);
      constexpr uint32_t idesc = umma_idesc_bf16(kMergeTile, kMergeTile, 1, 0);
      int nb_loaded = -1, bt_loads = 0, bt_frees = 0;
      int i = 0;   // A tiles consumed
      for (int tile = t_begin; tile < t_end; ++i, ++tile) {
        const int nb = tile / k_tiles, slot = i % kMpASlots, buf = i & 1;
        if (nb != nb_loaded) {
          if (bt_loads > 0) {
            // the MMAs that read the previous B^T must have completed
            umma_commit(bt_free);
            if (!mbar_wait(bt_free, bt_frees & 1, ab)) break;
            ++bt_frees;
          }
          load_bt(nb);
          if (!mbar_wait(bt_full, bt_loads & 1, ab)) break;
          ++bt_loads;
          nb_loaded = nb;
        }
        if (!mbar_wait(a_full(slot), (i / kMpASlots) & 1, ab)) break;
        if (!mbar_wait(tmem_empty(buf), ((i >> 1) & 1) ^ 1, ab)) {
          ++i;   // this tile's copy has landed
          break;
        }
        tc_fence_after_sync();
        const uint32_t d = tmem + static_cast<uint32_t>(buf * kMergeTile);
#pragma unroll
        for (int c = 0; c < S::kChunks; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sw128_desc(base + S::kBtOff + c * 16384 + kk * 2048, 8192, 1024);
            const uint64_t bd = sw128_desc(base + S::kAOff + slot * S::kOpBytes + c * 16384 + kk * 32, 16, 1024);
            umma_bf16(d, ad, bd, idesc, (c | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(a_empty(slot));
        umma_commit(tmem_full(buf));
        // refill the slot for the tile kMpASlots ahead once these MMAs have read it
        if (t_begin + loaded < t_end) {
          if (!mbar_wait(a_empty(slot), (i / kMpASlots) & 1, ab)) {
            ++i;
            break;
          }
          load_a(t_begin + loaded, slot);
          ++loaded;
        }
      }
      // after a wait ran out: let the A copies still in flight land
      for (int q = i; q < loaded; ++q) mbar_wait(a_full(q % kMpASlots), (q / kMpASlots) & 1, ab, false);
      // every MMA issued here has completed before TMEM is released
      umma_commit(drain);
      mbar_wait(drain, 0, ab, false);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warps 0-7 finish the CTA's even tiles (accumulator 0),
    // warps 8-15 its odd ones (accumulator 1); in each half, thread (quarter, q)
    // takes row i of the tile, columns 64*q .. 64*q+63: one whole NF4 block, so
    // one block table serves 64 elements
    const int half = warp >> 3, hw = warp & 7;
    const int quarter = hw & 3, q = hw >> 2;
    const int i = quarter * 32 + lane;
    // each warp stores its own 32 x 64 box (its TMEM rows, its 64 columns)
    // from two 4 KB stagings of its own, so no barrier spans the warps
    const uint32_t my_stage = base + S::kStageOff + static_cast<uint32_t>(warp) * 8192u;
    const int kblocks = p.K >> 6;
    // codes (32 B) and absmax of tile `tile` for this thread, zero outside the matrix
    auto fetch = [&](int tile, uint4& ca, uint4& cb, float& am) {
      ca = make_uint4(0u, 0u, 0u, 0u);
      cb = ca;
      am = 0.0f;
      if (tile >= t_end) return;
      const int n = (tile / k_tiles) * kMergeTile + i, k = (tile % k_tiles) * kMergeTile + 64 * q;
      if (n >= p.N || k >= p.K) return;
      const uint8_t* src = p.packed + static_cast<int64_t>(n) * (p.K / 2) + k / 2;
      ca = ldg_nc_v4(src);
      cb = ldg_nc_v4(src + 16);
      am = ldg_nc_f32(p.absmax + static_cast<int64_t>(n) * kblocks + (k >> 6));
    };
    // this half's tiles are t_begin + half, + 2, ...; the next two are fetched ahead
    uint4 c0a, c0b, c1a, c1b, c2a, c2b;
    float a0, a1, a2;
    fetch(t_begin + half, c0a, c0b, a0);
    fetch(t_begin + half + 2, c1a, c1b, a1);
    for (int j = 0, tile = t_begin + half; tile < t_end; ++j, tile += 2) {
      fetch(tile + 4, c2a, c2b, a2);
      // a warp whose wait ran out only skips the work
      const bool ok = __all_sync(0xffffffffu, mbar_wait(tmem_full(half), j & 1, ab));
      const int sb = j & 1;   // this warp's staging, last stored two of its tiles ago
      if (lane == 0) tma_store_wait_read_le1();
      __syncwarp();
      if (ok) {
        tc_fence_after_sync();
        const Nf4BlockTable tab = nf4_block_table(a0);
        const uint32_t words[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
        // staging: this warp's [32 rows][64 columns], 128-byte rows, 128-byte swizzle
        const uint32_t row = my_stage + static_cast<uint32_t>(sb) * 4096u + static_cast<uint32_t>(lane) * 128u;
        const uint32_t tacc = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>(half * kMergeTile + 64 * q);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t v[32];
          tmem_ld32(tacc + 32u * hh, v);
          tmem_ld_wait();
          if (hh == 1) {
            // both column halves are in registers: the accumulator may be overwritten
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty(half));
          }
#pragma unroll
          for (int wq = 0; wq < 4; ++wq) {
            const uint4 wd = nf4_expand8(words[4 * hh + wq], tab);   // elements 32hh + 8wq .. +7 of the block
            const uint32_t pr[4] = {wd.x, wd.y, wd.z, wd.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float w0 = __uint_as_float(pr[e] << 16), w1 = __uint_as_float(pr[e] & 0xFFFF0000u);
              o[e] = pack_bf16x2(fmaf(p.s, __uint_as_float(v[8 * wq + 2 * e]), w0),
                                 fmaf(p.s, __uint_as_float(v[8 * wq + 2 * e + 1]), w1));
            }
            const uint32_t chunk = static_cast<uint32_t>(4 * hh + wq) ^ (static_cast<uint32_t>(lane) & 7u);
            st_shared_v4(row + (chunk << 4), make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0 && ok) {
        // boxes wholly outside the matrix are not stored
        const int nr = (tile / k_tiles) * kMergeTile + quarter * 32, kc = (tile % k_tiles) * kMergeTile + 64 * q;
        if (nr < p.N && kc < p.K) {
          tma_store_2d(&map_out, my_stage + static_cast<uint32_t>(sb) * 4096u, kc, nr);
          tma_store_commit();
        }
      }
      c0a = c1a;
      c0b = c1b;
      a0 = a1;
      c1a = c2a;
      c1b = c2b;
      a1 = a2;
    }
    if (lane == 0) tma_store_wait_all();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 256);
  }
}

template <int RP>
cudaError_t launch_merge_rp(const CUtensorMap& map_out, const MergeParams& mp, cudaStream_t stream) {
  auto kern = lora_merge_kernel<RP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MergeSmem<RP>::kBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((mp.K + kMergeTile - 1) / kMergeTile, (mp.N + kMergeTile - 1) / kMergeTile);
  LaunchScope scope(kKindMerge, stream);
  kern<<<grid, kMergeThreads, MergeSmem<RP>::kBytes, stream>>>(map_out, mp);
  return cudaGetLastError();
}

template <int RP>
cudaError_t launch_merge_persistent_rp(const CUtensorMap (&maps)[3], const MergeParams& mp, cudaStream_t stream) {
  auto kern = lora_merge_persistent_kernel<RP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MergePSmem<RP>::kBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int k_tiles = (mp.K + kMergeTile - 1) / kMergeTile;
  const int tiles = k_tiles * ((mp.N + kMergeTile - 1) / kMergeTile);
  const int grid = std::min(tiles, sms);
  LaunchScope scope(kKindMerge, stream);
  kern<<<grid, kMpThreads, MergePSmem<RP>::kBytes, stream>>>(maps[0], maps[1], maps[2], mp, k_tiles, tiles);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_nf4(const uint8_t* packed, const float* absmax, int N, int K, const uint16_t* A,
                             const uint16_t* B, int r, float s, uint16_t* out, int* status,
                             cudaStream_t stream) {
  CUtensorMap map_out;
  if (!make_bf16_map_sw128(&map_out, out, static_cast<uint64_t>(K), static_cast<uint64_t>(N), 64, kMergeTile))
    return cudaErrorInvalidValue;
  MergeParams mp;
  mp.packed = packed;
  mp.absmax = absmax;
  mp.A = A;
  mp.B = B;
  mp.N = N;
  mp.K = K;
  mp.r = r;
  mp.s = s;
  mp.a_vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0 && r % 8 == 0) ? 1 : 0;
  mp.b_vec = (reinterpret_cast<uintptr_t>(B) % 16 == 0) ? 1 : 0;
  mp.status = status;
  if (mp.a_vec && mp.b_vec) {
    // A^T and B^T tiles by TMA: rows of A are r * 2 bytes (a multiple of 16 when r % 8 == 0)
    CUtensorMap maps[3];
    if (!make_tensor_map_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, static_cast<uint64_t>(K),
                            static_cast<uint64_t>(N), static_cast<uint64_t>(K) * 2, 64, 32,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, static_cast<uint64_t>(r),
                            static_cast<uint64_t>(K), static_cast<uint64_t>(r) * 2, 64, kMergeTile,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, static_cast<uint64_t>(N),
                            static_cast<uint64_t>(r), static_cast<uint64_t>(N) * 2, 64, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    if (r <= 64) return launch_merge_persistent_rp<64>(maps, mp, stream);
    return launch_merge_persistent_rp<128>(maps, mp, stream);
  }
  if (r <= 64) return launch_merge_rp<64>(map_out, mp, stream);
  return launch_merge_rp<128>(map_out, mp, stream);
}

}  // namespace qlora
