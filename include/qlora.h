/*
 * qlora.h -- C ABI of the fused NF4-QLoRA linear layer for NVIDIA B300 (sm_103a).
 *
 * The layer: a frozen base weight W [d_out, d_in] stored in 4-bit NF4, a
 * trainable low-rank pair A [d_in, r], B [r, d_out], scale s, no dropout, no bias:
 *
 *     Y  = X . W_deq^T + s . (X . A) . B
 *     dX = dY . W_deq + s . (dY . B^T) . A^T
 *     dA = s . X^T . (dY . B^T)
 *     dB = s . (X . A)^T . dY          (no gradient for the frozen W)
 *
 * Sources on the Unsloth pages:
 *   - the fused Linear -> LoRA_A -> LoRA_B -> Add chain, "UnSloth加速原理：CUDA内核融合与内存优化",
 *     section "内核融合" (its ReLU between LoRA_A and LoRA_B is not LoRA and is not computed);
 *   - A in R^{d_in x r}, B in R^{r x d_out}: same page, section "LoRA张量的紧凑布局";
 *   - lora_dropout=0, bias="none", load_in_4bit (NF4): same page, section "内核融合";
 *   - the hand-written backward: "解锁 AI 潜能：Unsloth 的算法奥秘与实现全解析", section
 *     "Triton 编写的高效内核", and "Unsloth性能实测：比传统方法快2倍真的吗？", section 3.2;
 *   - s = alpha/r or alpha/sqrt(r) (rank-stabilised): "Unsloth更新日志解读：新功能带来的实际收益",
 *     section 2.1.  The caller passes s itself.
 *
 * NF4 format (the pages name NF4 only; this is the plainest reading): the
 * 16-level NF4 table of QLoRA (Dettmers et al., 2023, Appendix E); blocks of
 * 64 consecutive elements of the row-major weight; one fp32 absmax per block
 * (no second-level quantisation); codes q = nearest level of fl32(w/absmax),
 * ties to the lower index, all-zero blocks -> code 7 (0.0) and absmax 0; two
 * codes per byte, FIRST element in the HIGH nibble.  Dequantised value:
 * bf16_rne(fl32(code[q] * absmax)).
 *
 * Conventions for every call:
 *   - bf16 tensors are passed as `uint16_t*` bit patterns; all tensors are
 *     dense, row-major, contiguous, in DEVICE memory owned by the caller;
 *   - every device pointer must be 16-byte aligned (QLORA_ERR_ALIGN);
 *   - calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream); the library allocates no device memory; scratch comes
 *     from the caller's `workspace`;
 *   - argument errors return a non-OK status and launch nothing; a failed
 *     launch returns QLORA_ERR_CUDA and qlora_last_cuda_error() gives the
 *     cudaError_t value;
 *   - every device-side wait is bounded (about one second); a wait that runs
 *     out records QLORA_ERR_TIMEOUT in a device status word read by
 *     qlora_device_status(); the kernel then returns without finishing;
 *   - the library caches, per device, the device addresses of its own device
 *     variables (the status word, the no-allocation scratch array); do not
 *     keep using a loaded library across cudaDeviceReset() or a reset of the
 *     primary context, which moves them.
 */
#ifndef QLORA_H_
#define QLORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qlora_status {
  QLORA_OK = 0,
  QLORA_ERR_NULL = 1,         /* a required pointer is NULL */
  QLORA_ERR_SHAPE = 2,        /* a size is negative, zero where not allowed, or too large */
  QLORA_ERR_ALIGN = 3,        /* a device pointer is not 16-byte aligned */
  QLORA_ERR_UNSUPPORTED = 4,  /* d_in % 64 != 0, d_out % 8 != 0, r outside [1, 256] ([1, 128] for the merge) */
  QLORA_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed; see qlora_last_cuda_error() */
  QLORA_ERR_TIMEOUT = 6,      /* a bounded device-side wait ran out (see qlora_device_status) */
  QLORA_ERR_WORKSPACE = 7,    /* workspace NULL or smaller than qlora_workspace_bytes() */
  QLORA_ERR_INTERNAL = 8      /* a kernel found its shared-memory layout does not fit its launch
                                 (recorded in the device status word; nothing was computed) */
} qlora_status;

struct CUstream_st;
typedef struct CUstream_st* qlora_stream_t; /* identical to cudaStream_t */

/* Human-readable name of a status code (static string, never NULL). */
const char* qlora_status_string(qlora_status status);

/* cudaError_t value of the most recent failing CUDA call made by this library
 * on the calling thread (0 if none). */
int qlora_last_cuda_error(void);

/* Host copy of the 16 NF4 levels the kernels use, ascending (for checks). */
void qlora_nf4_codebook(float out[16]);

/* Synchronises the current device, then reads the library's device status
 * word into *code (a qlora_status; QLORA_OK if no kernel recorded an error)
 * and clears it when `clear` is non-zero.  Returns QLORA_ERR_CUDA if the
 * synchronisation or the read fails. */
qlora_status qlora_device_status(int* code, int clear);

/* Launch accounting for measurement tools.
 * qlora_profile_enable(1): from now on every kernel the library launches is
 * bracketed by two CUDA events recorded on the launching stream (events are
 * created on first use and reused; no device memory is allocated).
 * qlora_profile_collect: waits for the recorded events, writes for each kernel
 * kind launched since the last collect its name (static string), total
 * device milliseconds and launch count, returns the number of kinds written
 * (at most max_kinds), and clears the records.  Returns -1 on a CUDA error.
 * qlora_launch_count: kernels launched by this library since it was loaded. */
qlora_status qlora_profile_enable(int enable);
int qlora_profile_collect(const char** names, float* total_ms, int* launches, int max_kinds);
int64_t qlora_launch_count(void);

/* Test hook for the error path of the bounded device waits (off by default;
 * an interface addition of this library, with no counterpart on the pages).
 * The next `launches` launches of the fused main kernel (the forward Y for
 * more than 16 tokens, the backward dX) load no token operand: no stage
 * completes, the waits run out after about one second, the kernel records
 * QLORA_ERR_TIMEOUT in the status word (qlora_device_status), releases its
 * tensor memory and returns with nothing in flight; its output is left
 * unwritten or partly written.  0 switches the hook off.  Returns
 * QLORA_ERR_SHAPE for a negative count. */
qlora_status qlora_debug_stall_main_launches(int launches);

/*
 * NF4 quantisation of a bf16 weight (offline; once per weight).
 *   W       [n_out, n_in] bf16, read.
 *   packed  [n_out * n_in / 2] bytes, written (2 codes per byte, high nibble first).
 *   absmax  [n_out * n_in / 64] fp32, written (block b = elements 64b..64b+63
 *           of the row-major flattening).
 * Requires n_out >= 1, n_in >= 64, n_in % 64 == 0.  W must be finite
 * (non-finite inputs give unspecified codes).  Bit-exact with the format
 * above: division is IEEE correctly rounded, boundaries are exact midpoints.
 * Pages: "UnSloth加速原理：CUDA内核融合与内存优化", section "内核融合" (load_in_4bit).
 */
qlora_status qlora_quantize_nf4(const uint16_t* W, int64_t n_out, int64_t n_in,
                                uint8_t* packed, float* absmax, qlora_stream_t stream);

/*
 * NF4 dequantisation: W_out[i] = bf16_rne(fl32(code[q_i] * absmax[i / 64])).
 *   packed, absmax as produced by qlora_quantize_nf4 (read);
 *   W_out  [n_out, n_in] bf16, written.
 * Requires n_out >= 1, n_in >= 64, n_in % 64 == 0.  Bit-exact.
 * The fused kernels dequantise with the same per-block table, so their
 * weight operand equals this output bit for bit.
 */
qlora_status qlora_dequant_nf4(const uint8_t* packed, const float* absmax,
                               int64_t n_out, int64_t n_in, uint16_t* W_out,
                               qlora_stream_t stream);

/*
 * The block absmax stored in 8 bits (row f4, "double quantisation"; QLoRA,
 * Dettmers et al. 2023, section 3, which the pages' load_in_4bit stands on:
 * "UnSloth加速原理：CUDA内核融合与内存优化", section 内核融合).  Groups of 256
 * consecutive block absmax values (the last may be shorter); per group g, with
 * c_g its largest value,
 *   scale2[g] = fl32(c_g / 255)  (0 when c_g == 0),
 *   q8[i]     = the integer nearest fl32(absmax[i] / scale2[g]), ties to even,
 *               at most 255 (0 when scale2[g] == 0),
 * and back: absmax'[i] = fl32(q8[i] * scale2[g]).  Storage per weight element:
 * 0.5 + 1/64 + 1/4096 bytes instead of 0.5 + 1/16.  The layer calls take the
 * fp32 absmax': expand it (qlora_dequant_absmax_dq, n_blocks * 4 bytes of
 * scratch) before a call; everything downstream (the NF4 dequantisation, the
 * fused kernels) is unchanged.
 *   absmax  [n_blocks] fp32 (read by _quantize, written by _dequant);
 *   q8      [n_blocks] bytes; scale2 [ceil(n_blocks / 256)] fp32.
 * Requires n_blocks >= 1; all pointers 16-byte aligned.  Asynchronous on `stream`.
 */
qlora_status qlora_quantize_absmax_dq(const float* absmax, int64_t n_blocks, uint8_t* q8, float* scale2,
                                      qlora_stream_t stream);
qlora_status qlora_dequant_absmax_dq(const uint8_t* q8, const float* scale2, int64_t n_blocks, float* absmax,
                                     qlora_stream_t stream);


/*
 * Merged 16-bit weight: the adapter folded into the base weight,
 *   W_out[n, k] = bf16_rne(fma(s, (A . B)[k, n], W_deq[n, k]))
 * with W_deq the qlora_dequant_nf4 expansion (bit for bit) and (A . B) the
 * rank-r product accumulated in fp32 on the tensor core.
 *   packed, absmax  the NF4 weight [d_out, d_in] as produced by qlora_quantize_nf4 (read);
 *   A  [d_in, r] bf16 and B [r, d_out] bf16, row-major (read; no alignment needed);
 *   W_out [d_out, d_in] bf16, written.
 * Re-quantising the merged weight to NF4 is qlora_quantize_nf4 on W_out.
 * Requires d_in % 64 == 0, d_out % 8 == 0, 1 <= r <= 128; packed, absmax and
 * W_out 16-byte aligned.  Asynchronous on `stream`; a device-side wait that
 * runs out sets the status word (qlora_device_status).
 * Pages: "这不是“魔法”是把Unsloth的底层优化逻辑榨干了用", section 4
 * (save_pretrained_merged, "merged_16bit").
 */
qlora_status qlora_merge_nf4(const uint8_t* packed, const float* absmax, int64_t d_out, int64_t d_in,
                             const uint16_t* A, const uint16_t* B, int32_t r, float s, uint16_t* W_out,
                             qlora_stream_t stream);

/*
 * SwiGLU gate of the MLP block, between the stacked gate/up projection and the
 * down projection (the pages fuse the MLP into their forward: "Unsloth性能实测：
 * 比传统方法快2倍真的吗？", section 2.2; SwiGLU is among the fused transformer
 * operators of "UnSloth加速原理：CUDA内核融合与内存优化", section "在ms-swift中的角色"):
 *   h[m, j] = bf16_rne(silu(g) * u),  g = gu[m, j], u = gu[m, d_ff + j],
 *   silu(x) = x / (1 + e^-x), fp32 arithmetic.
 *   gu [M, 2*d_ff] bf16 (gate columns, then up columns), read;  h [M, d_ff] bf16, written.
 * Requires M >= 0 (0 launches nothing), d_ff % 8 == 0; gu and h 16-byte aligned.
 */
qlora_status qlora_swiglu_fwd(const uint16_t* gu, int64_t M, int64_t d_ff, uint16_t* h, qlora_stream_t stream);

/*
 * Its backward, written in the layout of gu (the dY of the stacked projection):
 *   dgu[m, j]        = bf16_rne(dh * u * sigma(g) * (1 + g * (1 - sigma(g))))   (d/dg)
 *   dgu[m, d_ff + j] = bf16_rne(dh * silu(g))                                   (d/du)
 *   gu [M, 2*d_ff] and dh [M, d_ff] bf16, read;  dgu [M, 2*d_ff] bf16, written.
 * Same requirements as qlora_swiglu_fwd (gu, dh, dgu 16-byte aligned).
 */
qlora_status qlora_swiglu_bwd(const uint16_t* gu, const uint16_t* dh, int64_t M, int64_t d_ff, uint16_t* dgu,
                              qlora_stream_t stream);

/* Bytes of scratch qlora_linear_fwd / qlora_linear_bwd need for this shape
 * (0 if the shape is unsupported).  The same workspace serves both calls. */
size_t qlora_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int32_t r);

/*
 * Forward:  Y = X . W_deq^T + s . T . B,   T = X . A   (T saved for the backward).
 *   X        [M, d_in]  bf16, read.
 *   packed, absmax: NF4 weight of shape [d_out, d_in] (qlora_quantize_nf4 layout), read.
 *   A        [d_in, r]  bf16, read.      B [r, d_out] bf16, read.
 *   s        LoRA scale (alpha/r or alpha/sqrt(r)).
 *   Y        [M, d_out] bf16, written (overwritten, never accumulated into).
 *   XA_save  [M, r]     fp32, written: T, needed by qlora_linear_bwd.
 *   workspace / workspace_bytes: caller scratch, >= qlora_workspace_bytes().
 * Requires M >= 0 (M == 0 launches nothing), d_in % 64 == 0, d_out % 8 == 0,
 * 1 <= r <= 256.  Accuracy: fp32 accumulation of bf16 products; the LoRA term
 * enters the tensor-core accumulator as bf16(s*T) x B.  For 1..16 tokens with
 * d_in % 256 == 0 the weight is streamed by a separate kernel that multiplies
 * bf16(level[q]) by X and applies each block's absmax to the block sum in fp32:
 * the same result up to the rounding of the weight (both within 2^-9 of
 * level[q] * absmax).
 */
qlora_status qlora_linear_fwd(const uint16_t* X, int64_t M, int64_t d_in, int64_t d_out,
                              const uint8_t* packed, const float* absmax,
                              const uint16_t* A, const uint16_t* B, int32_t r, float s,
                              uint16_t* Y, float* XA_save,
                              void* workspace, size_t workspace_bytes,
                              qlora_stream_t stream);

/*
 * Forward that allocates nothing: the same computation and outputs as
 * qlora_linear_fwd, without the workspace arguments.  (An interface addition
 * of this library; the Unsloth pages have no counterpart.)
 *
 * For callers that cannot hand the layer a workspace: a process whose device
 * memory belongs to another allocator, a loop that must not allocate after
 * start-up, or glue code that only holds the layer's own tensors.  Its
 * scratch is a fixed 8 MiB device array inside this library, which every GPU
 * that loads the library keeps for the life of the process.
 *   - Needs M * rp * 2 bytes of that array, plus d_in * rp * 2 bytes when
 *     r % 8 != 0 (a zero-padded copy of A), rp = 64 * ceil(r / 64), each part
 *     rounded up to 1 KiB; larger shapes return QLORA_ERR_WORKSPACE and launch
 *     nothing.  What is left of the array holds the split-work counters and
 *     partial tiles; with too little left the kernels fall back to whole tiles.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - All calls share the array: calls whose GPU work overlaps (other
 *     streams, unordered threads) race on it.  Everything a call reads from
 *     it is written earlier in the same call, so nothing needs clearing.
 * Other arguments, requirements and errors as qlora_linear_fwd.
 */
qlora_status qlora_linear_fwd_noalloc(const uint16_t* X, int64_t M, int64_t d_in, int64_t d_out,
                                      const uint8_t* packed, const float* absmax,
                                      const uint16_t* A, const uint16_t* B, int32_t r, float s,
                                      uint16_t* Y, float* XA_save, qlora_stream_t stream);

/*
 * Backward (the hand-written gradients; W is frozen, so there is no dW):
 *   G  = dY . B^T
 *   dX = dY . W_deq + s . G . A^T      [M, d_in]  bf16, written; may be NULL to skip
 *   dA = s . X^T . G                   [d_in, r]  fp32, written (overwritten)
 *   dB = s . T^T . dY                  [r, d_out] fp32, written (overwritten)
 *   X [M, d_in], dY [M, d_out] bf16, read; XA_saved [M, r] fp32 = T from the
 *   forward, read; packed/absmax/A/B/r/s as in the forward.
 * M == 0 writes dA = dB = 0.  Reductions over M are deterministic (fixed
 * order, no atomics on data).  Pages: "Unsloth性能实测：比传统方法快2倍真的吗？",
 * section 3.2 (LoRA gradients injected directly, no autograd graph).
 */
qlora_status qlora_linear_bwd(const uint16_t* X, const uint16_t* dY,
                              int64_t M, int64_t d_in, int64_t d_out,
                              const uint8_t* packed, const float* absmax,
                              const uint16_t* A, const uint16_t* B, int32_t r, float s,
                              const float* XA_saved,
                              uint16_t* dX, float* dA, float* dB,
                              void* workspace, size_t workspace_bytes,
                              qlora_stream_t stream);

/*
 * Stacked projections of one input with separate low-rank blocks ("target
 * modules" of one activation: q/k/v, gate/up; "UnSloth加速原理：CUDA内核融合与内存优化",
 * section 内核融合).  n_groups projections are one layer whose weight rows are
 * stacked along d_out (group g owns output features [sum_{i<g} group_d_out[i],
 * sum_{i<=g} group_d_out[i])) and whose low-rank part is block-diagonal:
 *   A [d_in, r] with group g in columns [g*group_rank, (g+1)*group_rank),
 *   B [r, d_out] with group g's block in those rows and its own columns, zero
 *     elsewhere (the zeros are read: G = dY.B^T runs over all of B),
 *   r = n_groups * group_rank (zero-padded columns of A give zero rows of dB).
 * The forward's low-rank term and dB touch only the diagonal blocks: each
 * output tile adds its own group's T columns times its B block, and dB is
 * written only in the diagonal blocks (the off-diagonal blocks are left as
 * they were).  Everything else -- Y, T, dX (summed over the groups), dA --
 * is qlora_linear_fwd / _bwd with the same A and B.
 * Requires 1 <= n_groups <= 8, group_rank % 64 == 0, r <= 256, every
 * group_d_out but the last a multiple of 128, and qlora_linear_fwd's other
 * requirements with d_out = sum group_d_out; the workspace is
 * qlora_workspace_bytes(M, d_in, d_out, r).  group_d_out is a host array.
 */
qlora_status qlora_linear_fwd_grouped(const uint16_t* X, int64_t M, int64_t d_in, int32_t n_groups,
                                      const int64_t* group_d_out, int32_t group_rank, const uint8_t* packed,
                                      const float* absmax, const uint16_t* A, const uint16_t* B, float s,
                                      uint16_t* Y, float* XA_save, void* workspace, size_t workspace_bytes,
                                      qlora_stream_t stream);

qlora_status qlora_linear_bwd_grouped(const uint16_t* X, const uint16_t* dY, int64_t M, int64_t d_in,
                                      int32_t n_groups, const int64_t* group_d_out, int32_t group_rank,
                                      const uint8_t* packed, const float* absmax, const uint16_t* A,
                                      const uint16_t* B, float s, const float* XA_saved, uint16_t* dX, float* dA,
                                      float* dB, void* workspace, size_t workspace_bytes, qlora_stream_t stream);


/*
 * SwiGLU MLP block with the gate fused into the layers' epilogues.
 *
 *     gu = X . W_gu_deq^T + s_gu . (X . A_gu) . B_gu      (gate and up projections, one layer)
 *     h  = silu(g) * u,   silu(x) = x / (1 + e^-x)
 *     Y  = h . W_d_deq^T + s_d . (h . A_d) . B_d          (down projection)
 *
 * The pages fuse the MLP of the transformer block into their forward
 * ("Unsloth性能实测：比传统方法快2倍真的吗？", section 2.2) and name SwiGLU among the
 * fused transformer operators ("UnSloth加速原理：CUDA内核融合与内存优化", section
 * "在ms-swift中的角色").  Here the gate costs no pass of its own: the gate/up
 * layer's epilogue writes h beside gu, and the down layer's backward epilogue
 * turns its input gradient dh into dgu (the gate's backward) without storing dh.
 *
 * Layout of the gate/up layer (d_in -> 2*d_ff, d_ff % 64 == 0): its weight rows,
 * the columns of B_gu and the columns of gu are INTERLEAVED in 64-row chunks,
 *     [gate 0..63 | up 0..63 | gate 64..127 | up 64..127 | ...],
 * so that every 128-feature output tile holds matching gate and up features.
 * Quantise the interleaved bf16 weight with qlora_quantize_nf4 (NF4 blocks lie
 * within a row, so its codes are the separate weights' codes, rows permuted).
 * Rounding: gu, h, dh and dgu are rounded to bf16 at the points where an
 * unfused block stores them, and the gate's arithmetic is fp32, so the fused
 * block computes what the unfused one (qlora_linear_* + qlora_swiglu_*) does.
 */

/* Forward of the interleaved gate/up layer: gu [M, 2*d_ff] (the layer's Y) and
 * h [M, d_ff], both bf16, written; XA_save [M, r] fp32 written (T for the
 * backward).  Other arguments and requirements as qlora_linear_fwd with
 * d_out = 2*d_ff; d_ff % 64 == 0.  For 1..16 tokens the gate is a separate
 * elementwise pass after the weight-stream kernel. */
qlora_status qlora_linear_fwd_swiglu(const uint16_t* X, int64_t M, int64_t d_in, int64_t d_ff,
                                     const uint8_t* packed, const float* absmax,
                                     const uint16_t* A, const uint16_t* B, int32_t r, float s,
                                     uint16_t* gu, uint16_t* h, float* XA_save,
                                     void* workspace, size_t workspace_bytes, qlora_stream_t stream);

/* Backward of the down layer (d_ff -> d_out) of the block: as qlora_linear_bwd
 * with X = h, except that the layer's input gradient dh is not stored;
 * instead dgu [M, 2*d_ff] bf16 (interleaved like gu) is written,
 *   dgu[gate f] = dh * u * sigma(g) * (1 + g * (1 - sigma(g))),  dgu[up f] = dh * silu(g),
 * from gu [M, 2*d_ff] (read, the forward's).  dA, dB as in qlora_linear_bwd. */
qlora_status qlora_linear_bwd_swiglu(const uint16_t* h, const uint16_t* dY, int64_t M, int64_t d_ff,
                                     int64_t d_out, const uint8_t* packed, const float* absmax,
                                     const uint16_t* A, const uint16_t* B, int32_t r, float s,
                                     const float* XA_saved, const uint16_t* gu, uint16_t* dgu,
                                     float* dA, float* dB, void* workspace, size_t workspace_bytes,
                                     qlora_stream_t stream);

/* Workspace for qlora_swiglu_mlp_fwd / _bwd (the larger of the two layers'); 0 if unsupported. */
size_t qlora_swiglu_mlp_workspace_bytes(int64_t M, int64_t d_model, int64_t d_ff, int32_t r_gu, int32_t r_d);

/* The whole block forward: qlora_linear_fwd_swiglu, then the down layer.
 *   X [M, d_model] read; Y [M, d_model] written; gu [M, 2*d_ff], h [M, d_ff],
 *   T_gu [M, r_gu], T_d [M, r_d] written (saved for the backward).
 *   gate/up layer: gu_packed, gu_absmax (interleaved [2*d_ff, d_model] weight),
 *   A_gu [d_model, r_gu], B_gu [r_gu, 2*d_ff] (interleaved columns), s_gu;
 *   down layer: d_packed, d_absmax ([d_model, d_ff] weight), A_d [d_ff, r_d],
 *   B_d [r_d, d_model], s_d.
 * Requires d_model % 64 == 0, d_ff % 64 == 0, ranks in [1, 256]. */
qlora_status qlora_swiglu_mlp_fwd(const uint16_t* X, int64_t M, int64_t d_model, int64_t d_ff,
                                  const uint8_t* gu_packed, const float* gu_absmax, const uint16_t* A_gu,
                                  const uint16_t* B_gu, int32_t r_gu, float s_gu,
                                  const uint8_t* d_packed, const float* d_absmax, const uint16_t* A_d,
                                  const uint16_t* B_d, int32_t r_d, float s_d,
                                  uint16_t* Y, uint16_t* gu, uint16_t* h, float* T_gu, float* T_d,
                                  void* workspace, size_t workspace_bytes, qlora_stream_t stream);

/* The whole block backward: qlora_linear_bwd_swiglu (down layer, writes dgu),
 * then the gate/up layer's backward with dY = dgu.
 *   X, dY [M, d_model] read; gu, h, T_gu, T_d from the forward, read;
 *   dgu [M, 2*d_ff] bf16: caller scratch, written; dX [M, d_model] bf16 written
 *   (may be NULL to skip); dA_gu, dB_gu, dA_d, dB_d fp32 written (overwritten).
 * Same layer arguments and requirements as qlora_swiglu_mlp_fwd. */
qlora_status qlora_swiglu_mlp_bwd(const uint16_t* X, const uint16_t* dY, int64_t M, int64_t d_model, int64_t d_ff,
                                  const uint8_t* gu_packed, const float* gu_absmax, const uint16_t* A_gu,
                                  const uint16_t* B_gu, int32_t r_gu, float s_gu,
                                  const uint8_t* d_packed, const float* d_absmax, const uint16_t* A_d,
                                  const uint16_t* B_d, int32_t r_d, float s_d,
                                  const uint16_t* gu, const uint16_t* h, const float* T_gu, const float* T_d,
                                  uint16_t* dgu, uint16_t* dX, float* dA_gu, float* dB_gu, float* dA_d,
                                  float* dB_d, void* workspace, size_t workspace_bytes, qlora_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_H_ */
