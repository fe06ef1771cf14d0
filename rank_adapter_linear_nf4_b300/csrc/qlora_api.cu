// qlora_api.cu -- the C ABI (include/qlora.h): argument validation, status
// codes, the device status word, and launch sequencing on the caller's stream.
#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>
#include <cuda_runtime.h>

#include "qlora.h"
#include "kernels.h"

namespace {

thread_local int g_last_cuda_error = 0;

// Device status word: bounded device-side waits that run out write here.
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
// Per-device cache of the status word's address; filled under g_status_mu so
// that threads making their first call on a device at once do not race.
std::mutex g_status_mu;
std::atomic<int*> g_status_ptr[kMaxDevices] = {};

qlora_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return QLORA_ERR_CUDA;
}

// Device address of the status word for the current device.
qlora_status status_word(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return QLORA_ERR_UNSUPPORTED;
  int* word = g_status_ptr[dev].load(std::memory_order_acquire);
  if (word == nullptr) {
    std::lock_guard<std::mutex> lock(g_status_mu);
    word = g_status_ptr[dev].load(std::memory_order_relaxed);
    if (word == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_device_status);
      if (e != cudaSuccess) return cuda_fail(e);
      word = static_cast<int*>(p);
      g_status_ptr[dev].store(word, std::memory_order_release);
    }
  }
  *out = word;
  return QLORA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest sizes the kernels index with 32-bit coordinates.
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

qlora_status check_codec_shape(int64_t n_out, int64_t n_in) {
  if (n_out < 1 || n_in < 1) return QLORA_ERR_SHAPE;
  if (n_in % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  if (n_out > kMaxDim || n_in > kMaxDim || n_out * n_in / 64 > kMaxDim * 8) return QLORA_ERR_SHAPE;
  return QLORA_OK;
}

qlora_status check_layer(int64_t M, int64_t d_in, int64_t d_out, int32_t r) {
  if (M < 0 || d_in < 1 || d_out < 1) return QLORA_ERR_SHAPE;
  if (M > kMaxDim || d_in > kMaxDim || d_out > kMaxDim) return QLORA_ERR_SHAPE;
  if (d_in % 64 != 0 || d_out % 8 != 0 || r < 1 || r > qlora::kMaxRank) return QLORA_ERR_UNSUPPORTED;
  return QLORA_OK;
}

qlora::LayerDims dims_of(int64_t M, int64_t d_in, int64_t d_out, int32_t r, float s) {
  qlora::LayerDims d;
  d.M = static_cast<int>(M);
  d.K = static_cast<int>(d_in);
  d.N = static_cast<int>(d_out);
  d.r = r;
  d.rp = qlora::padded_rank(r);
  d.s = s;
  return d;
}

// ---------------------------------------------------------------- launch accounting

std::atomic<int64_t> g_launches{0};
std::atomic<bool> g_profiling{false};

struct ProfRecord {
  int kind;
  cudaEvent_t begin, end;
};

std::mutex g_prof_mu;
std::vector<ProfRecord> g_records;     // recorded since the last collect
std::vector<cudaEvent_t> g_free_events;

const char* const kKindNames[qlora::kNumKernelKinds] = {
    "nf4_quantize", "nf4_dequant", "lora_pad_A", "lora_rows_T", "lora_rows_G",
    "lora_red_dA_dB", "lora_main_fwd", "lora_main_dX", "lora_merge", "lora_stream_fwd", "swiglu_fwd", "swiglu_bwd",
    "lora_stream_finish", "nf4_absmax_dq"};

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

namespace qlora {

void record_cuda_error(int cuda_error) { g_last_cuda_error = cuda_error; }

namespace {
std::atomic<int> g_debug_stall_launches{0};
}  // namespace

bool take_debug_stall() {
  int n = g_debug_stall_launches.load(std::memory_order_relaxed);
  while (n > 0) {
    if (g_debug_stall_launches.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) return true;
  }
  return false;
}

int* device_status_word(int* cuda_error) {
  int* word = nullptr;
  const qlora_status st = status_word(&word);
  if (cuda_error != nullptr) *cuda_error = (st == QLORA_OK) ? 0 : g_last_cuda_error;
  return st == QLORA_OK ? word : nullptr;
}

LaunchScope::LaunchScope(int k, cudaStream_t s) : kind(k), stream(s), slot(-1) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_profiling.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  ProfRecord r{k, take_event(), take_event()};
  if (r.begin == nullptr || r.end == nullptr) return;
  if (cudaEventRecord(r.begin, s) != cudaSuccess) return;
  slot = static_cast<int>(g_records.size());
  g_records.push_back(r);
}

LaunchScope::~LaunchScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaEventRecord(g_records[slot].end, stream);
}

}  // namespace qlora

extern "C" {

qlora_status qlora_profile_enable(int enable) {
  g_profiling.store(enable != 0);
  return QLORA_OK;
}

int qlora_profile_collect(const char** names, float* total_ms, int* launches, int max_kinds) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  float ms[qlora::kNumKernelKinds] = {0};
  int cnt[qlora::kNumKernelKinds] = {0};
  bool failed = false;
  for (const ProfRecord& r : g_records) {
    float t = 0.0f;
    if (cudaEventSynchronize(r.end) != cudaSuccess ||
        cudaEventElapsedTime(&t, r.begin, r.end) != cudaSuccess)
      failed = true;
    ms[r.kind] += t;
    cnt[r.kind] += 1;
    g_free_events.push_back(r.begin);
    g_free_events.push_back(r.end);
  }
  g_records.clear();
  if (failed) return -1;
  int n = 0;
  for (int k = 0; k < qlora::kNumKernelKinds && n < max_kinds; ++k) {
    if (cnt[k] == 0) continue;
    if (names) names[n] = kKindNames[k];
    if (total_ms) total_ms[n] = ms[k];
    if (launches) launches[n] = cnt[k];
    ++n;
  }
  return n;
}

int64_t qlora_launch_count(void) { return g_launches.load(); }

qlora_status qlora_debug_stall_main_launches(int launches) {
  if (launches < 0) return QLORA_ERR_SHAPE;
  qlora::g_debug_stall_launches.store(launches);
  return QLORA_OK;
}


const char* qlora_status_string(qlora_status status) {
  switch (status) {
    case QLORA_OK: return "QLORA_OK";
    case QLORA_ERR_NULL: return "QLORA_ERR_NULL: a required pointer is NULL";
    case QLORA_ERR_SHAPE: return "QLORA_ERR_SHAPE: invalid or too large size";
    case QLORA_ERR_ALIGN: return "QLORA_ERR_ALIGN: device pointer not 16-byte aligned";
    case QLORA_ERR_UNSUPPORTED:
      return "QLORA_ERR_UNSUPPORTED: need d_in % 64 == 0, d_out % 8 == 0, 1 <= r <= 128";
    case QLORA_ERR_CUDA: return "QLORA_ERR_CUDA: a CUDA call failed (qlora_last_cuda_error)";
    case QLORA_ERR_TIMEOUT: return "QLORA_ERR_TIMEOUT: a bounded device wait ran out";
    case QLORA_ERR_WORKSPACE: return "QLORA_ERR_WORKSPACE: workspace missing or too small";
    case QLORA_ERR_INTERNAL: return "QLORA_ERR_INTERNAL: a kernel's shared-memory layout did not fit";
  }
  return "unknown qlora_status";
}

int qlora_last_cuda_error(void) { return g_last_cuda_error; }

void qlora_nf4_codebook(float out[16]) {
  if (out != nullptr) qlora::nf4_levels_host(out);
}

qlora_status qlora_device_status(int* code, int clear) {
  if (code == nullptr) return QLORA_ERR_NULL;
  int* word = nullptr;
  qlora_status st = status_word(&word);
  if (st != QLORA_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  int v = 0;
  e = cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (clear) {
    e = cudaMemset(word, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  *code = v;
  return QLORA_OK;
}

qlora_status qlora_quantize_nf4(const uint16_t* W, int64_t n_out, int64_t n_in, uint8_t* packed,
                                float* absmax, qlora_stream_t stream) {
  qlora_status st = check_codec_shape(n_out, n_in);
  if (st != QLORA_OK) return st;
  if (!W || !packed || !absmax) return QLORA_ERR_NULL;
  if (!aligned16(W) || !aligned16(packed) || !aligned16(absmax)) return QLORA_ERR_ALIGN;
  cudaError_t e = qlora::launch_quantize_nf4(W, n_out * n_in, packed, absmax,
                                             reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_dequant_nf4(const uint8_t* packed, const float* absmax, int64_t n_out,
                               int64_t n_in, uint16_t* W_out, qlora_stream_t stream) {
  qlora_status st = check_codec_shape(n_out, n_in);
  if (st != QLORA_OK) return st;
  if (!packed || !absmax || !W_out) return QLORA_ERR_NULL;
  if (!aligned16(packed) || !aligned16(absmax) || !aligned16(W_out)) return QLORA_ERR_ALIGN;
  cudaError_t e = qlora::launch_dequant_nf4(packed, absmax, n_out * n_in, W_out,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_quantize_absmax_dq(const float* absmax, int64_t n_blocks, uint8_t* q8, float* scale2,
                                      qlora_stream_t stream) {
  if (n_blocks < 1 || n_blocks > kMaxDim * 8) return QLORA_ERR_SHAPE;
  if (!absmax || !q8 || !scale2) return QLORA_ERR_NULL;
  if (!aligned16(absmax) || !aligned16(q8) || !aligned16(scale2)) return QLORA_ERR_ALIGN;
  cudaError_t e = qlora::launch_quantize_absmax_dq(absmax, n_blocks, q8, scale2, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_dequant_absmax_dq(const uint8_t* q8, const float* scale2, int64_t n_blocks, float* absmax,
                                     qlora_stream_t stream) {
  if (n_blocks < 1 || n_blocks > kMaxDim * 8) return QLORA_ERR_SHAPE;
  if (!absmax || !q8 || !scale2) return QLORA_ERR_NULL;
  if (!aligned16(absmax) || !aligned16(q8) || !aligned16(scale2)) return QLORA_ERR_ALIGN;
  cudaError_t e = qlora::launch_dequant_absmax_dq(q8, scale2, n_blocks, absmax, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_merge_nf4(const uint8_t* packed, const float* absmax, int64_t d_out, int64_t d_in,
                             const uint16_t* A, const uint16_t* B, int32_t r, float s, uint16_t* W_out,
                             qlora_stream_t stream) {
  if (d_out < 1 || d_in < 1) return QLORA_ERR_SHAPE;
  const int64_t max_dim = (int64_t(1) << 31) - 1;
  if (d_out > max_dim || d_in > max_dim || (d_out + 127) / 128 > 65535) return QLORA_ERR_SHAPE;
  if (d_in % 64 != 0 || d_out % 8 != 0 || r < 1 || r > 128) return QLORA_ERR_UNSUPPORTED;
  if (!packed || !absmax || !A || !B || !W_out) return QLORA_ERR_NULL;
  if (!aligned16(packed) || !aligned16(absmax) || !aligned16(W_out)) return QLORA_ERR_ALIGN;
  int cuda_error = 0;
  int* status = qlora::device_status_word(&cuda_error);
  if (status == nullptr) return cuda_fail(static_cast<cudaError_t>(cuda_error));
  cudaError_t e = qlora::launch_merge_nf4(packed, absmax, static_cast<int>(d_out), static_cast<int>(d_in), A, B, r,
                                          s, W_out, status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

namespace {
qlora_status check_swiglu(int64_t M, int64_t d_ff) {
  if (M < 0 || d_ff < 1) return QLORA_ERR_SHAPE;
  if (d_ff > (int64_t(1) << 30) || (M > 0 && M > (int64_t(1) << 40) / d_ff)) return QLORA_ERR_SHAPE;
  if (d_ff % 8 != 0) return QLORA_ERR_UNSUPPORTED;
  return QLORA_OK;
}
}  // namespace

qlora_status qlora_swiglu_fwd(const uint16_t* gu, int64_t M, int64_t d_ff, uint16_t* h, qlora_stream_t stream) {
  const qlora_status st = check_swiglu(M, d_ff);
  if (st != QLORA_OK) return st;
  if (M == 0) return QLORA_OK;
  if (!gu || !h) return QLORA_ERR_NULL;
  if (!aligned16(gu) || !aligned16(h)) return QLORA_ERR_ALIGN;
  cudaError_t e = qlora::launch_swiglu_fwd(gu, M, d_ff, h, false, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_swiglu_bwd(const uint16_t* gu, const uint16_t* dh, int64_t M, int64_t d_ff, uint16_t* dgu,
                              qlora_stream_t stream) {
  const qlora_status st = check_swiglu(M, d_ff);
  if (st != QLORA_OK) return st;
  if (M == 0) return QLORA_OK;
  if (!gu || !dh || !dgu) return QLORA_ERR_NULL;
  if (!aligned16(gu) || !aligned16(dh) || !aligned16(dgu)) return QLORA_ERR_ALIGN;
  cudaError_t e = qlora::launch_swiglu_bwd(gu, dh, M, d_ff, dgu, false, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

size_t qlora_workspace_bytes(int64_t M, int64_t d_in, int64_t d_out, int32_t r) {
  if (check_layer(M, d_in, d_out, r) != QLORA_OK) return 0;
  return qlora::workspace_bytes(dims_of(M, d_in, d_out, r, 1.0f));
}

qlora_status qlora_linear_fwd(const uint16_t* X, int64_t M, int64_t d_in, int64_t d_out,
                              const uint8_t* packed, const float* absmax, const uint16_t* A,
                              const uint16_t* B, int32_t r, float s, uint16_t* Y, float* XA_save,
                              void* workspace, size_t workspace_bytes, qlora_stream_t stream) {
  qlora_status st = check_layer(M, d_in, d_out, r);
  if (st != QLORA_OK) return st;
  if (!packed || !absmax || !A || !B) return QLORA_ERR_NULL;
  if (M == 0) return QLORA_OK;
  if (!X || !Y || !XA_save) return QLORA_ERR_NULL;
  if (!aligned16(X) || !aligned16(packed) || !aligned16(absmax) || !aligned16(A) ||
      !aligned16(B) || !aligned16(Y) || !aligned16(XA_save) || !aligned16(workspace))
    return QLORA_ERR_ALIGN;
  const qlora::LayerDims d = dims_of(M, d_in, d_out, r, s);
  if (workspace == nullptr || workspace_bytes < qlora::workspace_bytes(d)) return QLORA_ERR_WORKSPACE;
  int* status = nullptr;
  st = status_word(&status);
  if (st != QLORA_OK) return st;
  cudaError_t e = qlora::run_forward(d, X, packed, absmax, A, B, Y, XA_save,
                                     qlora::carve_workspace(d, workspace), status,
                                     reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_linear_bwd(const uint16_t* X, const uint16_t* dY, int64_t M, int64_t d_in,
                              int64_t d_out, const uint8_t* packed, const float* absmax,
                              const uint16_t* A, const uint16_t* B, int32_t r, float s,
                              const float* XA_saved, uint16_t* dX, float* dA, float* dB,
                              void* workspace, size_t workspace_bytes, qlora_stream_t stream) {
  qlora_status st = check_layer(M, d_in, d_out, r);
  if (st != QLORA_OK) return st;
  if (!packed || !absmax || !A || !B || !dA || !dB) return QLORA_ERR_NULL;
  if (!aligned16(packed) || !aligned16(absmax) || !aligned16(A) || !aligned16(B) ||
      !aligned16(dA) || !aligned16(dB))
    return QLORA_ERR_ALIGN;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    // empty sums: dA = dB = 0
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * static_cast<size_t>(d_in) * r, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, sizeof(float) * static_cast<size_t>(d_out) * r, cs);
    return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
  }
  if (!X || !dY || !XA_saved) return QLORA_ERR_NULL;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(XA_saved) || !aligned16(workspace) ||
      (dX != nullptr && !aligned16(dX)))
    return QLORA_ERR_ALIGN;
  const qlora::LayerDims d = dims_of(M, d_in, d_out, r, s);
  if (workspace == nullptr || workspace_bytes < qlora::workspace_bytes(d)) return QLORA_ERR_WORKSPACE;
  int* status = nullptr;
  st = status_word(&status);
  if (st != QLORA_OK) return st;
  cudaError_t e = qlora::run_backward(d, X, dY, packed, absmax, A, B, XA_saved, dX, dA, dB,
                                      qlora::carve_workspace(d, workspace), status, cs);
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- stacked projections, separate low-rank blocks

namespace {
// Group layout of a stacked layer; fills d_out and the kernels' LoraGroups.
qlora_status check_groups(int32_t n_groups, const int64_t* group_d_out, int32_t group_rank, int64_t* d_out,
                          qlora::LoraGroups* g) {
  if (group_d_out == nullptr) return QLORA_ERR_NULL;
  if (n_groups < 1 || n_groups > qlora::kMaxLoraGroups || group_rank < 1) return QLORA_ERR_UNSUPPORTED;
  if (group_rank % 64 != 0 || static_cast<int64_t>(n_groups) * group_rank > qlora::kMaxRank)
    return QLORA_ERR_UNSUPPORTED;
  int64_t end = 0;
  *g = qlora::LoraGroups{};
  g->n = n_groups;
  g->width = group_rank;
  for (int i = 0; i < n_groups; ++i) {
    if (group_d_out[i] < 1 || group_d_out[i] > kMaxDim) return QLORA_ERR_SHAPE;
    if (i + 1 < n_groups && group_d_out[i] % 128 != 0) return QLORA_ERR_UNSUPPORTED;
    end += group_d_out[i];
    if (end > kMaxDim) return QLORA_ERR_SHAPE;
    g->end[i] = static_cast<int>(end);
  }
  *d_out = end;
  return QLORA_OK;
}
}  // namespace

qlora_status qlora_linear_fwd_grouped(const uint16_t* X, int64_t M, int64_t d_in, int32_t n_groups,
                                      const int64_t* group_d_out, int32_t group_rank, const uint8_t* packed,
                                      const float* absmax, const uint16_t* A, const uint16_t* B, float s,
                                      uint16_t* Y, float* XA_save, void* workspace, size_t workspace_bytes,
                                      qlora_stream_t stream) {
  int64_t d_out = 0;
  qlora::LoraGroups groups;
  qlora_status st = check_groups(n_groups, group_d_out, group_rank, &d_out, &groups);
  if (st != QLORA_OK) return st;
  const int32_t r = n_groups * group_rank;
  st = check_layer(M, d_in, d_out, r);
  if (st != QLORA_OK) return st;
  if (!packed || !absmax || !A || !B) return QLORA_ERR_NULL;
  if (M == 0) return QLORA_OK;
  if (!X || !Y || !XA_save) return QLORA_ERR_NULL;
  if (!aligned16(X) || !aligned16(packed) || !aligned16(absmax) || !aligned16(A) || !aligned16(B) ||
      !aligned16(Y) || !aligned16(XA_save) || !aligned16(workspace))
    return QLORA_ERR_ALIGN;
  qlora::LayerDims d = dims_of(M, d_in, d_out, r, s);
  if (workspace == nullptr || workspace_bytes < qlora::workspace_bytes(d)) return QLORA_ERR_WORKSPACE;
  d.groups = groups;
  int* status = nullptr;
  st = status_word(&status);
  if (st != QLORA_OK) return st;
  cudaError_t e = qlora::run_forward(d, X, packed, absmax, A, B, Y, XA_save, qlora::carve_workspace(d, workspace),
                                     status, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_linear_bwd_grouped(const uint16_t* X, const uint16_t* dY, int64_t M, int64_t d_in,
                                      int32_t n_groups, const int64_t* group_d_out, int32_t group_rank,
                                      const uint8_t* packed, const float* absmax, const uint16_t* A,
                                      const uint16_t* B, float s, const float* XA_saved, uint16_t* dX, float* dA,
                                      float* dB, void* workspace, size_t workspace_bytes, qlora_stream_t stream) {
  int64_t d_out = 0;
  qlora::LoraGroups groups;
  qlora_status st = check_groups(n_groups, group_d_out, group_rank, &d_out, &groups);
  if (st != QLORA_OK) return st;
  const int32_t r = n_groups * group_rank;
  st = check_layer(M, d_in, d_out, r);
  if (st != QLORA_OK) return st;
  if (!packed || !absmax || !A || !B || !dA || !dB) return QLORA_ERR_NULL;
  if (!aligned16(packed) || !aligned16(absmax) || !aligned16(A) || !aligned16(B) || !aligned16(dA) ||
      !aligned16(dB))
    return QLORA_ERR_ALIGN;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * static_cast<size_t>(d_in) * r, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, sizeof(float) * static_cast<size_t>(d_out) * r, cs);
    return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
  }
  if (!X || !dY || !XA_saved) return QLORA_ERR_NULL;
  if (!aligned16(X) || !aligned16(dY) || !aligned16(XA_saved) || !aligned16(workspace) ||
      (dX != nullptr && !aligned16(dX)))
    return QLORA_ERR_ALIGN;
  qlora::LayerDims d = dims_of(M, d_in, d_out, r, s);
  if (workspace == nullptr || workspace_bytes < qlora::workspace_bytes(d)) return QLORA_ERR_WORKSPACE;
  d.groups = groups;
  int* status = nullptr;
  st = status_word(&status);
  if (st != QLORA_OK) return st;
  cudaError_t e = qlora::run_backward(d, X, dY, packed, absmax, A, B, XA_saved, dX, dA, dB,
                                      qlora::carve_workspace(d, workspace), status, cs);
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

// ---------------------------------------------------------------- SwiGLU MLP block, gate fused

qlora_status qlora_linear_fwd_swiglu(const uint16_t* X, int64_t M, int64_t d_in, int64_t d_ff,
                                     const uint8_t* packed, const float* absmax, const uint16_t* A,
                                     const uint16_t* B, int32_t r, float s, uint16_t* gu, uint16_t* h,
                                     float* XA_save, void* workspace, size_t workspace_bytes,
                                     qlora_stream_t stream) {
  if (d_ff < 1 || d_ff > kMaxDim / 2) return QLORA_ERR_SHAPE;
  if (d_ff % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  const int64_t d_out = 2 * d_ff;
  qlora_status st = check_layer(M, d_in, d_out, r);
  if (st != QLORA_OK) return st;
  if (!packed || !absmax || !A || !B) return QLORA_ERR_NULL;
  if (M == 0) return QLORA_OK;
  if (!X || !gu || !h || !XA_save) return QLORA_ERR_NULL;
  if (!aligned16(X) || !aligned16(packed) || !aligned16(absmax) || !aligned16(A) || !aligned16(B) ||
      !aligned16(gu) || !aligned16(h) || !aligned16(XA_save) || !aligned16(workspace))
    return QLORA_ERR_ALIGN;
  const qlora::LayerDims d = dims_of(M, d_in, d_out, r, s);
  if (workspace == nullptr || workspace_bytes < qlora::workspace_bytes(d)) return QLORA_ERR_WORKSPACE;
  int* status = nullptr;
  st = status_word(&status);
  if (st != QLORA_OK) return st;
  cudaError_t e = qlora::run_forward(d, X, packed, absmax, A, B, gu, XA_save, qlora::carve_workspace(d, workspace),
                                     status, reinterpret_cast<cudaStream_t>(stream), h);
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

qlora_status qlora_linear_bwd_swiglu(const uint16_t* h, const uint16_t* dY, int64_t M, int64_t d_ff,
                                     int64_t d_out, const uint8_t* packed, const float* absmax,
                                     const uint16_t* A, const uint16_t* B, int32_t r, float s,
                                     const float* XA_saved, const uint16_t* gu, uint16_t* dgu, float* dA,
                                     float* dB, void* workspace, size_t workspace_bytes, qlora_stream_t stream) {
  if (d_ff < 1 || d_ff > kMaxDim / 2) return QLORA_ERR_SHAPE;
  if (d_ff % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  qlora_status st = check_layer(M, d_ff, d_out, r);
  if (st != QLORA_OK) return st;
  if (!packed || !absmax || !A || !B || !dA || !dB) return QLORA_ERR_NULL;
  if (!aligned16(packed) || !aligned16(absmax) || !aligned16(A) || !aligned16(B) || !aligned16(dA) ||
      !aligned16(dB))
    return QLORA_ERR_ALIGN;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(float) * static_cast<size_t>(d_ff) * r, cs);
    if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, sizeof(float) * static_cast<size_t>(d_out) * r, cs);
    return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
  }
  if (!h || !dY || !XA_saved || !gu || !dgu) return QLORA_ERR_NULL;
  if (!aligned16(h) || !aligned16(dY) || !aligned16(XA_saved) || !aligned16(gu) || !aligned16(dgu) ||
      !aligned16(workspace))
    return QLORA_ERR_ALIGN;
  const qlora::LayerDims d = dims_of(M, d_ff, d_out, r, s);
  if (workspace == nullptr || workspace_bytes < qlora::workspace_bytes(d)) return QLORA_ERR_WORKSPACE;
  int* status = nullptr;
  st = status_word(&status);
  if (st != QLORA_OK) return st;
  cudaError_t e = qlora::run_backward(d, h, dY, packed, absmax, A, B, XA_saved, nullptr, dA, dB,
                                      qlora::carve_workspace(d, workspace), status, cs, gu, dgu);
  return e == cudaSuccess ? QLORA_OK : cuda_fail(e);
}

namespace {
qlora_status check_mlp(int64_t M, int64_t d_model, int64_t d_ff, int32_t r_gu, int32_t r_d) {
  if (d_ff < 1 || d_ff > kMaxDim / 2) return QLORA_ERR_SHAPE;
  if (d_ff % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  const qlora_status a = check_layer(M, d_model, 2 * d_ff, r_gu);
  return a != QLORA_OK ? a : check_layer(M, d_ff, d_model, r_d);
}
}  // namespace

size_t qlora_swiglu_mlp_workspace_bytes(int64_t M, int64_t d_model, int64_t d_ff, int32_t r_gu, int32_t r_d) {
  if (d_ff < 1 || d_ff > kMaxDim / 2 || d_ff % 64 != 0) return 0;
  const size_t a = qlora_workspace_bytes(M, d_model, 2 * d_ff, r_gu);
  const size_t b = qlora_workspace_bytes(M, d_ff, d_model, r_d);
  if (a == 0 || b == 0) return 0;
  return a > b ? a : b;
}

qlora_status qlora_swiglu_mlp_fwd(const uint16_t* X, int64_t M, int64_t d_model, int64_t d_ff,
                                  const uint8_t* gu_packed, const float* gu_absmax, const uint16_t* A_gu,
                                  const uint16_t* B_gu, int32_t r_gu, float s_gu, const uint8_t* d_packed,
                                  const float* d_absmax, const uint16_t* A_d, const uint16_t* B_d, int32_t r_d,
                                  float s_d, uint16_t* Y, uint16_t* gu, uint16_t* h, float* T_gu, float* T_d,
                                  void* workspace, size_t workspace_bytes, qlora_stream_t stream) {
  const qlora_status shape = check_mlp(M, d_model, d_ff, r_gu, r_d);
  if (shape != QLORA_OK) return shape;
  if (workspace == nullptr || workspace_bytes < qlora_swiglu_mlp_workspace_bytes(M, d_model, d_ff, r_gu, r_d))
    return QLORA_ERR_WORKSPACE;
  qlora_status st = qlora_linear_fwd_swiglu(X, M, d_model, d_ff, gu_packed, gu_absmax, A_gu, B_gu, r_gu, s_gu, gu,
                                            h, T_gu, workspace, workspace_bytes, stream);
  if (st != QLORA_OK) return st;
  return qlora_linear_fwd(h, M, d_ff, d_model, d_packed, d_absmax, A_d, B_d, r_d, s_d, Y, T_d, workspace,
                          workspace_bytes, stream);
}

qlora_status qlora_swiglu_mlp_bwd(const uint16_t* X, const uint16_t* dY, int64_t M, int64_t d_model, int64_t d_ff,
                                  const uint8_t* gu_packed, const float* gu_absmax, const uint16_t* A_gu,
                                  const uint16_t* B_gu, int32_t r_gu, float s_gu, const uint8_t* d_packed,
                                  const float* d_absmax, const uint16_t* A_d, const uint16_t* B_d, int32_t r_d,
                                  float s_d, const uint16_t* gu, const uint16_t* h, const float* T_gu,
                                  const float* T_d, uint16_t* dgu, uint16_t* dX, float* dA_gu, float* dB_gu,
                                  float* dA_d, float* dB_d, void* workspace, size_t workspace_bytes,
                                  qlora_stream_t stream) {
  const qlora_status shape = check_mlp(M, d_model, d_ff, r_gu, r_d);
  if (shape != QLORA_OK) return shape;
  if (workspace == nullptr || workspace_bytes < qlora_swiglu_mlp_workspace_bytes(M, d_model, d_ff, r_gu, r_d))
    return QLORA_ERR_WORKSPACE;
  qlora_status st = qlora_linear_bwd_swiglu(h, dY, M, d_ff, d_model, d_packed, d_absmax, A_d, B_d, r_d, s_d, T_d,
                                            gu, dgu, dA_d, dB_d, workspace, workspace_bytes, stream);
  if (st != QLORA_OK) return st;
  return qlora_linear_bwd(X, dgu, M, d_model, 2 * d_ff, gu_packed, gu_absmax, A_gu, B_gu, r_gu, s_gu, T_gu, dX,
                          dA_gu, dB_gu, workspace, workspace_bytes, stream);
}

}  // extern "C"
