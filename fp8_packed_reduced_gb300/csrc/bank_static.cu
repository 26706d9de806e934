// Bank refresh for callers that cannot allocate device memory.
//
// qkvp_quantize_bank needs a small caller-provided workspace for the
// per-layer partial maxima between its two kernels.  Some callers have no
// way to provide one: code that runs where every allocation goes through a
// pool it does not own (an embedding framework that forbids cudaMalloc
// outside its allocator), or a refresh issued from a context where an
// allocation could block or fail (inside a latency-critical optimizer step).
// qkvp_quantize_bank_static gives them the same refresh with the scratch in a
// fixed array of device memory that belongs to this library.
#include <cstring>
#include <mutex>

#include "kernels.cuh"

namespace {

// Largest bank this entry point refreshes in one call, in layers.
constexpr int kStaticMaxLayers = 128;
constexpr int kStaticScratchFloats = kStaticMaxLayers * qkvp::kBankAmaxBlocks;  // 16 KB

// The scratch: one partial maximum per (layer, block) of the amax kernel.
// Every GPU that loads this library holds these 16 KB until the process exits.
static __device__ __align__(256) float g_bank_scratch[kStaticScratchFloats];

// Device address of g_bank_scratch on the current device.  The name of the
// array in host code is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, once per device, with that device current.
float* scratch_on_current_device(cudaError_t* err) {
  static std::mutex mu;
  static float* addr[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_bank_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<float*>(p);
  }
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int qkvp_quantize_bank_static(int L, int D, int H, int d_qk, int d_v, const uint16_t* const* Wq,
                                         const uint16_t* const* Wk, const uint16_t* const* Wv, uint8_t* W8,
                                         uint8_t* W8T, float* w_scale, void* stream) {
  if (L < 1 || D < 1 || H < 1 || !Wq || !Wk || !Wv || !W8 || !W8T || !w_scale) return QKVP_ERR_INVALID_ARGUMENT;
  if (L > kStaticMaxLayers) return QKVP_ERR_UNSUPPORTED;   // beyond the fixed scratch
  if (D % 128 != 0 || D > 16384 || H > 128 || d_v != 128 || (d_qk != 64 && d_qk != 96 && d_qk != 128))
    return QKVP_ERR_UNSUPPORTED;
  qkvp::BankArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int l = 0; l < L; ++l) {
    if (!Wq[l] || !Wk[l] || !Wv[l]) return QKVP_ERR_INVALID_ARGUMENT;
    if (!aligned16(Wq[l]) || !aligned16(Wk[l]) || !aligned16(Wv[l])) return QKVP_ERR_MISALIGNED;
    a.Wq[l] = Wq[l];
    a.Wk[l] = Wk[l];
    a.Wv[l] = Wv[l];
  }
  if (!aligned16(W8) || !aligned16(W8T) || !aligned16(w_scale)) return QKVP_ERR_MISALIGNED;
  a.W8 = W8;
  a.W8T = W8T;
  a.w_scale = w_scale;
  a.L = L;
  a.D = D;
  a.Nq = H * d_qk;
  a.N = H * (2 * d_qk + d_v);
  cudaError_t e = cudaSuccess;
  float* partials = scratch_on_current_device(&e);
  if (partials == nullptr) return QKVP_ERR_CUDA;
  // The amax kernel writes every partial the quantise kernel reads, so the
  // scratch needs no clearing between calls.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (qkvp::launch_bank_amax(a, partials, s) != cudaSuccess) return QKVP_ERR_CUDA;
  if (qkvp::launch_bank_quant(a, partials, s) != cudaSuccess) return QKVP_ERR_CUDA;
  return QKVP_OK;
}
