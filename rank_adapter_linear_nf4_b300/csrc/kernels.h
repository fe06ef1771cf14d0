// kernels.h -- internal launch interface between the C ABI layer and the
// kernels (not part of the public API).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qlora {

// Kernel kinds for launch accounting (names in qlora_api.cu).
enum KernelKind : int {
  kKindQuantize = 0,
  kKindDequant,
  kKindPrep,
  kKindRowsT,
  kKindRowsG,
  kKindRed,
  kKindMainFwd,
  kKindMainDx,
  kKindMerge,
  kKindStream,
  kKindSwigluFwd,
  kKindSwigluBwd,
  kKindStreamFinish,
  kKindAbsmaxDq,
  kNumKernelKinds
};

// Brackets one kernel launch: counts it and, when profiling is enabled,
// records CUDA events around it on `stream`.
struct LaunchScope {
  LaunchScope(int kind, cudaStream_t stream);
  ~LaunchScope();
  int kind;
  cudaStream_t stream;
  int slot;
};

// Device address of the library's status word on the current device (nullptr
// on failure; *cuda_error then holds the cudaError_t value).
int* device_status_word(int* cuda_error);

// Makes qlora_last_cuda_error() report `cuda_error` on the calling thread.
void record_cuda_error(int cuda_error);

// Test hook (qlora_debug_stall_main_launches): true for each of the next n
// launches of the fused main kernel, which then loads no token operand.
bool take_debug_stall();

// NF4 codec (nf4_codec.cu).
cudaError_t launch_quantize_nf4(const uint16_t* W, int64_t n_elems, uint8_t* packed, float* absmax,
                                cudaStream_t stream);
// The block absmax in 8 bits (groups of kDqGroup blocks, one fp32 scale each)
// and back.
constexpr int kDqGroup = 256;
cudaError_t launch_quantize_absmax_dq(const float* absmax, int64_t n, uint8_t* q8, float* scale2,
                                      cudaStream_t stream);
cudaError_t launch_dequant_absmax_dq(const uint8_t* q8, const float* scale2, int64_t n, float* absmax,
                                     cudaStream_t stream);
cudaError_t launch_dequant_nf4(const uint8_t* packed, const float* absmax, int64_t n_elems,
                               uint16_t* W_out, cudaStream_t stream);
void nf4_levels_host(float out[16]);

// LoRA linear (lora_kernels.cu).
// Projections stacked along d_out whose low-rank parts stay separate (a
// block-diagonal B): group g owns output features [end[g-1], end[g]) and rank
// columns [g * width, (g + 1) * width).  With n == 0 the low-rank part is one
// dense block.
constexpr int kMaxLoraGroups = 8;
struct LoraGroups {
  int n = 0;
  int width = 0;                     // a multiple of 64
  int end[kMaxLoraGroups] = {};      // every end but the last a multiple of 128
};

struct LayerDims {
  int M;       // tokens
  int K;       // d_in
  int N;       // d_out
  int r;       // LoRA rank
  int rp;      // r padded to 64, 128 or 256 (padded_rank)
  float s;     // LoRA scale
  LoraGroups groups;   // separate low-rank blocks of stacked projections (forward Y and dB only)
};

// Largest LoRA rank of a layer call.
constexpr int kMaxRank = 256;

// The rank padded to a width the rank-r kernels are built for: 64, 128 or 256
// columns (the tensor-core N of their MMAs, the TMEM columns they allocate).
inline int padded_rank(int r) { return r <= 64 ? 64 : r <= 128 ? 128 : 256; }

// Workspace carve-up shared by the forward and the backward.
struct Workspace {
  uint16_t* a_pad;   // [K, rp]  A with zero columns r..rp-1 (used when r % 8 != 0)
  uint16_t* s_t;     // [M, rp]  bf16(s * X.A), zero-padded
  uint16_t* s_g;     // [M, rp]  bf16(s * dY.B^T), zero-padded
  // Split-remainder buffers of the main kernel (nullptr: whole tiles only).
  int* counters;         // pieces finished per split tile, zeroed by the rank-r kernel before it
  int counter_cap;
  float* partials;       // fp32 partial tiles
  size_t partial_bytes;
};
size_t workspace_bytes(const LayerDims& d);
// Counters the workspace holds: the main kernel's split tiles (one per SM) or
// the token-stream kernel's 64-row panels, whichever is more.
int counter_slots(const LayerDims& d);
// Bytes of partial tiles the main kernel, or for at most kStreamMaxTokens
// tokens the token-stream kernel, uses at most for these dimensions.
size_t split_partial_bytes(const LayerDims& d);
Workspace carve_workspace(const LayerDims& d, void* base);

// The SwiGLU gate fused into a layer's epilogue (rows of W and columns of the
// output interleaved in 64-row chunks, gate then up): the gate/up layer's
// forward also writes h (h != nullptr); the down layer's backward writes dgu
// from its dX and gu instead of storing dX (dgu != nullptr).
struct GateIo {
  uint16_t* h = nullptr;
  const uint16_t* gu = nullptr;
  uint16_t* dgu = nullptr;
};

// gate_h: nullptr, or h [M, N/2] for a gate/up layer with interleaved rows.
cudaError_t run_forward(const LayerDims& d, const uint16_t* X, const uint8_t* packed,
                        const float* absmax, const uint16_t* A, const uint16_t* B, uint16_t* Y,
                        float* XA, const Workspace& ws, int* status, cudaStream_t stream,
                        uint16_t* gate_h = nullptr);

// Forward for at most kStreamMaxTokens tokens as a stream of the NF4 weight
// (lora_stream.cu): the stream kernel, then a finishing kernel; it needs
// stream_partial_bytes(d, sms) of partial slots in the workspace.
constexpr int kStreamMaxTokens = 16;
// SMs the token-stream kernel leaves to the rank-r kernel before it (one
// 128-row tile, a cluster of at most 8 CTAs), which it overlaps.
constexpr int kStreamReservedSms = 8;
int stream_counter_slots(const LayerDims& d);
size_t stream_partial_bytes(const LayerDims& d, int sms);
bool stream_applies(const LayerDims& d, const Workspace& ws, int sms);
// T = X . A and bf16(s*T) for at most kStreamMaxTokens tokens (lora_xa_small.cu).
cudaError_t launch_xa_small(const LayerDims& d, const uint16_t* X, const uint16_t* A, int a_cols, float* XA,
                            const Workspace& ws, int* status, cudaStream_t stream);
cudaError_t launch_stream_fwd(const LayerDims& d, const uint16_t* X, const uint8_t* packed, const float* absmax,
                              const uint16_t* B, const Workspace& ws, uint16_t* Y, int* status, int sms,
                              cudaStream_t stream);

// Tensor map over a row-major bf16 [rows, cols] matrix, 128-byte swizzle.
bool make_bf16_map_sw128(CUtensorMap* m, const void* gaddr, uint64_t cols, uint64_t rows, uint32_t box_cols,
                         uint32_t box_rows);

// 2-D tensor map over a row-major [outer, inner] array (row_bytes apart).
bool make_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* gaddr, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

// SwiGLU gate of the MLP block (swiglu.cu): h = silu(g) * u from the stacked
// gate/up output gu [rows, 2*d_ff], and its backward into dgu (same layout).
// interleaved: gu's columns in 64-column chunks [gate 0..63 | up 0..63 | gate 64..127 | ...]
// instead of [gate | up] (d_ff % 64 == 0).
cudaError_t launch_swiglu_fwd(const uint16_t* gu, int64_t rows, int64_t d_ff, uint16_t* h, bool interleaved,
                              cudaStream_t stream);
cudaError_t launch_swiglu_bwd(const uint16_t* gu, const uint16_t* dh, int64_t rows, int64_t d_ff, uint16_t* dgu,
                              bool interleaved, cudaStream_t stream);

// Merged weight bf16(W_deq + s . (A . B)^T) (lora_merge.cu).
cudaError_t launch_merge_nf4(const uint8_t* packed, const float* absmax, int N, int K, const uint16_t* A,
                             const uint16_t* B, int r, float s, uint16_t* out, int* status,
                             cudaStream_t stream);

// gate_gu / gate_dgu: nullptr, or (for the down layer of a SwiGLU block, K = d_ff)
// gu [M, 2K] of the forward and dgu [M, 2K] written in place of dX.
cudaError_t run_backward(const LayerDims& d, const uint16_t* X, const uint16_t* dY,
                         const uint8_t* packed, const float* absmax, const uint16_t* A,
                         const uint16_t* B, const float* XA, uint16_t* dX, float* dA, float* dB,
                         const Workspace& ws, int* status, cudaStream_t stream,
                         const uint16_t* gate_gu = nullptr, uint16_t* gate_dgu = nullptr);

}  // namespace qlora
