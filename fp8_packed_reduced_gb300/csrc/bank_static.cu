// Bank refresh for callers that cannot allocate device memory.
//
// qkvp_quantize_bank needs a small caller-provided workspace for the
// counters and per-layer maxima its kernel shares between blocks.  Some
// callers have no way to provide one: code that runs where every allocation
// goes through a pool it does not own (an embedding framework that forbids
// cudaMalloc outside its allocator), or a refresh issued from a context where
// an allocation could block or fail (inside a latency-critical optimizer
// step).  qkvp_quantize_bank_static gives them the same refresh with the
// scratch in a fixed array of device memory that belongs to this library.
#include <cstring>
#include <mutex>

#include "kernels.cuh"

namespace {

// Largest bank this entry point refreshes in one call, in layers (the
// capacity of the per-layer arrays of qkvp::BankSync).
constexpr int kStaticMaxLayers = qkvp::kMaxLayers;

// The scratch: a status word (first error code, kernel id) in its first 256
// bytes, then the refresh kernel's counters.  2 KB; every GPU that loads
// this library holds it until the process exits.
constexpr size_t kStaticStatusBytes = 256;
constexpr size_t kStaticScratchBytes = 2048;
static_assert(kStaticStatusBytes + sizeof(qkvp::BankSync) <= kStaticScratchBytes, "scratch too small");
static __device__ __align__(256) unsigned char g_bank_scratch[kStaticScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the CUDA context current on this thread (0 if unavailable).
// A context that is destroyed and created again (cudaDeviceReset, or a host
// framework resetting the device) gets a new id.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_bank_scratch in the current device's context.  The
// name of the array in host code is only a host-side stand-in, so the address
// is looked up with cudaGetSymbolAddress with that device current, once per
// context (cached with the context's id and looked up again when it changes).
unsigned char* scratch_on_current_device(cudaError_t* err) {
  static std::mutex mu;
  static unsigned char* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
    // (this also makes the device's primary context current if no context is yet)
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_bank_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned char*>(p);
    ctx_of[dev] = current_context_id();
  }
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int qkvp_quantize_bank_static(int L, int D, int H, int d_qk, int d_v, const uint16_t* const* Wq,
                                         const uint16_t* const* Wk, const uint16_t* const* Wv, uint8_t* W8,
                                         uint8_t* W8T, float* w_scale, void* stream) {
  // the checks of qkvp_quantize_bank, in the same order, with the array's
  // capacity in place of the workspace size
  const qkvp_dims d{1, D, H, d_qk, d_v};
  if (L < 1 || !Wq || !Wk || !Wv || !W8 || !W8T || !w_scale) return QKVP_ERR_INVALID_ARGUMENT;
  const int rc = qkvp::check_dims(&d);
  if (rc != QKVP_OK) return rc;
  if (L > kStaticMaxLayers) return QKVP_ERR_UNSUPPORTED;   // beyond the fixed scratch
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
  unsigned char* scratch = scratch_on_current_device(&e);
  if (scratch == nullptr) return QKVP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernel leaves its counters at zero, but a call stopped by an error
  // may not have: clear the status word and the counters first (a memset of
  // the library's own array, no allocation).
  if (cudaMemsetAsync(scratch, 0, kStaticStatusBytes + sizeof(qkvp::BankSync), s) != cudaSuccess)
    return QKVP_ERR_CUDA;
  qkvp::mark(s);
  const qkvp::DevStatus st{reinterpret_cast<int*>(scratch), 2000000000ull};
  if (qkvp::launch_bank_refresh(a, reinterpret_cast<qkvp::BankSync*>(scratch + kStaticStatusBytes), st, s) !=
      cudaSuccess)
    return QKVP_ERR_CUDA;
  qkvp::mark(s);
  return QKVP_OK;
}
