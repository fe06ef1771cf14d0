// qlora_noalloc.cu -- a forward entry point that allocates nothing.
//
// qlora_linear_fwd needs a caller-provided workspace.  Some callers have no way
// to provide one at the point where they run the layer: a host runtime whose
// device memory is owned by another allocator (a stray cudaMalloc there
// would fragment or overrun its pool), a latency-critical loop that must not
// allocate after start-up, or glue code that only sees the layer's own
// tensors.  For them, qlora_linear_fwd_noalloc runs the same forward with its
// scratch in a fixed device array that is part of this library's image.
//
// The array costs kNoAllocScratchBytes of device memory on every GPU that
// loads the library, for the life of the process.  All calls share it, so
// calls whose GPU work overlaps (different streams, or threads without
// ordering between them) race on it; serialise them on one stream.  Every
// byte a call reads from the array is written earlier in the same call, so
// the contents left by the previous call never need clearing.
#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "kernels.h"
#include "qlora.h"

namespace {

// 8 MiB: enough for M * rp * 2 bytes (plus d_in * rp * 2 when r % 8 != 0) with
// rp = 64*ceil(r/64), e.g. M = 16384 tokens at r = 128, or M = 16384 tokens and
// d_in = 14336 at r = 100.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

size_t round_up_1k(size_t x) { return (x + 1023) & ~static_cast<size_t>(1023); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device.  The host-side
// name of the array is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" qlora_status qlora_linear_fwd_noalloc(const uint16_t* X, int64_t M, int64_t d_in,
                                                 int64_t d_out, const uint8_t* packed,
                                                 const float* absmax, const uint16_t* A,
                                                 const uint16_t* B, int32_t r, float s, uint16_t* Y,
                                                 float* XA_save, qlora_stream_t stream) {
  if (M < 0 || d_in < 1 || d_out < 1) return QLORA_ERR_SHAPE;
  const int64_t max_dim = (int64_t(1) << 31) - 1;
  if (M > max_dim || d_in > max_dim || d_out > max_dim) return QLORA_ERR_SHAPE;
  if (d_in % 64 != 0 || d_out % 8 != 0 || r < 1 || r > 128) return QLORA_ERR_UNSUPPORTED;
  if (!packed || !absmax || !A || !B) return QLORA_ERR_NULL;
  if (M == 0) return QLORA_OK;
  if (!X || !Y || !XA_save) return QLORA_ERR_NULL;
  if (!aligned16(X) || !aligned16(packed) || !aligned16(absmax) || !aligned16(A) || !aligned16(B) ||
      !aligned16(Y) || !aligned16(XA_save))
    return QLORA_ERR_ALIGN;

  qlora::LayerDims d;
  d.M = static_cast<int>(M);
  d.K = static_cast<int>(d_in);
  d.N = static_cast<int>(d_out);
  d.r = r;
  d.rp = qlora::padded_rank(r);
  d.s = s;
  // the forward reads and writes bf16(s*T) [M, rp] and, only for ranks whose
  // rows are not 16-byte multiples (r % 8 != 0), a zero-padded copy of A [d_in, rp]
  const size_t a_pad_bytes = (d.r % 8 != 0) ? round_up_1k(static_cast<size_t>(d.K) * d.rp * 2) : 0;
  const size_t s_t_bytes = round_up_1k(static_cast<size_t>(d.M) * d.rp * 2);
  if (a_pad_bytes + s_t_bytes > kNoAllocScratchBytes) return QLORA_ERR_WORKSPACE;

  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    qlora::record_cuda_error(static_cast<int>(e));
    return QLORA_ERR_CUDA;
  }
  int cuda_error = 0;
  int* status = qlora::device_status_word(&cuda_error);
  if (status == nullptr) return QLORA_ERR_CUDA;

  qlora::Workspace ws;
  ws.a_pad = a_pad_bytes != 0 ? static_cast<uint16_t*>(scratch) : nullptr;
  ws.s_t = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(scratch) + a_pad_bytes);
  ws.s_g = nullptr;   // backward only
  // what is left of the array holds the counters and partial tiles of the
  // main kernel and the token-stream kernel; without them the main kernel
  // takes whole tiles only
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    qlora::record_cuda_error(static_cast<int>(e));
    return QLORA_ERR_CUDA;
  }
  const int n_counters = std::max(sms, qlora::stream_counter_slots(d));
  const size_t counter_bytes = round_up_1k(static_cast<size_t>(n_counters) * sizeof(int));
  const size_t used = a_pad_bytes + s_t_bytes;
  ws.counters = nullptr;
  ws.counter_cap = 0;
  ws.partials = nullptr;
  ws.partial_bytes = 0;
  if (sms > 0 && used + counter_bytes < kNoAllocScratchBytes) {
    uint8_t* rest = static_cast<uint8_t*>(scratch) + used;
    ws.counters = reinterpret_cast<int*>(rest);
    ws.counter_cap = n_counters;
    ws.partials = reinterpret_cast<float*>(rest + counter_bytes);
    ws.partial_bytes = kNoAllocScratchBytes - used - counter_bytes;
  }
  e = qlora::run_forward(d, X, packed, absmax, A, B, Y, XA_save, ws, status,
                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    qlora::record_cuda_error(static_cast<int>(e));
    return QLORA_ERR_CUDA;
  }
  return QLORA_OK;
}
