// nf4_lut.cuh -- the library's NF4 code table and its dequantisation of one
// 64-element block through a per-block table held in registers.
//
// Format (the Unsloth pages name NF4 only -- "UnSloth加速原理：CUDA内核融合与内存优化",
// section "内核融合", load_in_4bit): the 16 NF4 levels of QLoRA (Dettmers et al.,
// 2023, Appendix E), one fp32 absmax per 64 consecutive elements, two codes
// per byte with the first element in the high nibble.  Dequantised value of
// code q in a block with absmax a: bf16_rne(fl32(level[q] * a)).
#pragma once

#include <cstdint>
#include "ptx.cuh"

namespace qlora {

// NF4 levels, ascending (QLoRA, Appendix E).  Host copy; the device copy
// below holds the same values.
constexpr float kNF4LevelsHost[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

static __constant__ float c_nf4_level[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

// Per-block table: the 16 dequantised bf16 values split into byte planes.
// lo[j] holds the low bytes of entries 4j..4j+3, hi[j] their high bytes.
struct Nf4BlockTable {
  uint32_t lo[4];
  uint32_t hi[4];
};

__device__ __forceinline__ Nf4BlockTable nf4_block_table(float absmax) {
  uint32_t pair[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // one fp32 multiply per level, rounded to nearest-even bf16
    const float e0 = __fmul_rn(c_nf4_level[2 * i], absmax);
    const float e1 = __fmul_rn(c_nf4_level[2 * i + 1], absmax);
    pair[i] = pack_bf16x2(e0, e1);          // entry 2i in the low half
  }
  Nf4BlockTable t;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    t.lo[j] = prmt(pair[2 * j], pair[2 * j + 1], 0x6420u);
    t.hi[j] = prmt(pair[2 * j], pair[2 * j + 1], 0x7531u);
  }
  return t;
}

// Four table lookups: each selector nibble is a 4-bit code; output byte k is
// plane byte of the code in nibble k.  Bit 3 of a code picks the upper half
// of the table (entries 8..15).
__device__ __forceinline__ uint32_t nf4_lookup4(const uint32_t (&plane)[4], uint32_t idx3,
                                                uint32_t sel_half) {
  const uint32_t low8 = prmt(plane[0], plane[1], idx3);
  const uint32_t high8 = prmt(plane[2], plane[3], idx3);
  return prmt(low8, high8, sel_half);
}

// Eight consecutive elements (one 32-bit word of packed codes, elements in
// memory order 0..7) -> eight bf16 values, element 0 in the lowest 16 bits.
// In the little-endian word, element 2i sits in the high nibble of byte i and
// element 2i+1 in its low nibble.
__device__ __forceinline__ uint4 nf4_expand8(uint32_t w, const Nf4BlockTable& t) {
  const uint32_t idx3 = w & 0x77777777u;                             // code & 7 per nibble
  const uint32_t half = ((w >> 1) & 0x44444444u) | 0x32103210u;      // nibble k -> k + 4*bit3
  uint4 out;
  {
    const uint32_t lo = nf4_lookup4(t.lo, idx3, half);   // bytes: e1, e0, e3, e2
    const uint32_t hi = nf4_lookup4(t.hi, idx3, half);
    out.x = prmt(lo, hi, 0x4051u);                       // {e0, e1}
    out.y = prmt(lo, hi, 0x6273u);                       // {e2, e3}
  }
  {
    const uint32_t i2 = idx3 >> 16, h2 = half >> 16;
    const uint32_t lo = nf4_lookup4(t.lo, i2, h2);       // bytes: e5, e4, e7, e6
    const uint32_t hi = nf4_lookup4(t.hi, i2, h2);
    out.z = prmt(lo, hi, 0x4051u);                       // {e4, e5}
    out.w = prmt(lo, hi, 0x6273u);                       // {e6, e7}
  }
  return out;
}

}  // namespace qlora
