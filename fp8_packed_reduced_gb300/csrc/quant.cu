// Bandwidth-bound quantisation kernels:
//   bank refresh  (amax per layer, then codes in both layouts, one launch)
//   x amax        (per-tensor amax of the activations)
//   x quantise    (codes of x, token-major)
//   RoPE table, and the timeout self-test kernel.
#include <algorithm>
#include <atomic>

#include "kernels.cuh"

namespace qkvp {

// ---------------------------------------------------------------------------
// Per-tensor amax of a bf16 tensor: one partial maximum per block.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float absmax_bf16x8(uint4 w) {
  float m = 0.f;
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(bf16_lo(u[i])));
    m = fmaxf(m, fabsf(bf16_hi(u[i])));
  }
  return m;
}

// x: n16 groups of 8 bf16 (16 bytes) followed by `tail` (< 8) bf16 values.
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint16_t* __restrict__ x, int64_t n16, int tail,
                                                         float* __restrict__ partials) {
  __shared__ float red[32];
  const uint4* p = reinterpret_cast<const uint4*>(x);
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 7 * stride < n16; i += 8 * stride) {  // eight independent loads in flight
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldg(p + i + j * stride);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, absmax_bf16x8(v[j]));
  }
  for (; i < n16; i += stride) m = fmaxf(m, absmax_bf16x8(__ldg(p + i)));
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail)
    m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[n16 * 8 + threadIdx.x]) << 16)));
  m = block_max(m, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

cudaError_t launch_amax_bf16(const uint16_t* x, int64_t n, float* partials, int blocks, cudaStream_t s) {
  amax_bf16_kernel<<<blocks, 256, 0, s>>>(x, n / 8, static_cast<int>(n % 8), partials);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bank refresh in one launch.  The refresh is a list of work items over the
// 128-row x 128-column tiles of all layers (layer by layer): items [0, U)
// take the amax of tile i, items [U, 2U) convert tile i - U into both code
// layouts.  Blocks claim items in order from a counter, so every amax item
// is held by a running block before the first conversion item is handed
// out: a block that waits for its layer's amax waits only on running blocks
// that never wait themselves.  The launch therefore needs no co-residency
// and may share the GPU with any other kernel.  An amax item folds its
// tile's maximum into the layer's word (a max reduction on the bit pattern,
// exact for non-negative floats) and then counts itself done; the block whose
// count completes the layer publishes the layer's scale (before it can wait
// on anything itself), and a conversion item waits (bounded) for that one
// word, then converts its tile, read again (from L2 for banks that fit
// there).  The last block out leaves the counters at zero for the next call.
// ---------------------------------------------------------------------------
__device__ __forceinline__ const uint16_t* bank_row(const BankArgs& a, int l, int n) {
  if (n < a.Nq) return a.Wq[l] + static_cast<int64_t>(n) * a.D;
  if (n < 2 * a.Nq) return a.Wk[l] + static_cast<int64_t>(n - a.Nq) * a.D;
  return a.Wv[l] + static_cast<int64_t>(n - 2 * a.Nq) * a.D;
}

// Transpose of a 4 x 4 byte block held as four row words: out[c] = bytes
// (r0[c], r1[c], r2[c], r3[c]).
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3, uint32_t (&out)[4]) {
  const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r0, r1, 0x7362);   // (r0c0 r1c0 r0c1 r1c1), (.. c2 .. c3)
  const uint32_t t2 = __byte_perm(r2, r3, 0x5140), t3 = __byte_perm(r2, r3, 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

// 16-byte read-only load with an L2 eviction-priority policy (createpolicy).
__device__ __forceinline__ uint4 ldg_hint(const uint4* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

constexpr int kBankThreads = 256;
constexpr int kBankWarps = kBankThreads / 32;

// Reductions without a returned value: max, and add with release semantics
// (the thread's earlier writes and reductions are visible before the add).
__device__ __forceinline__ void red_max_u32(unsigned int* p, unsigned int v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Add that returns the old value, with acquire and release semantics.
__device__ __forceinline__ unsigned int atom_add_acq_rel_u32(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_release_u32(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The count of an amax item of layer l returned `old` (acquire: every other
// item's maximum of the layer is visible); if it completed the layer, the
// layer's scale goes to w_scale and, released, to the published word.
__device__ __forceinline__ void bank_publish_if_last(const BankArgs& a, BankSync* sy, int l, unsigned int old,
                                                     unsigned int tpl) {
  if (old != tpl - 1) return;
  const float s = scale_from_amax(__uint_as_float(ld_relaxed_u32(&sy->amax[l])));
  a.w_scale[l] = s;
  st_release_u32(&sy->scale[l], __float_as_uint(s));   // s > 0: non-zero means published
}

// Tile of 128 bank rows x 128 columns.  Warp w, lane 16 h + j owns rows
// n0 + 16 w + 8 h + i (i < 8) and columns d0 + 8 j .. + 7: each load
// instruction of a half-warp reads one row's 256 contiguous bytes (two whole
// 128-byte lines).  Rows at or past N read nothing.
__device__ __forceinline__ void bank_load_tile(const BankArgs& a, int l, int n0, int d0, uint4 (&u)[8]) {
  const int w = threadIdx.x >> 5, h = (threadIdx.x >> 4) & 1, j = threadIdx.x & 15;
  const int nb = n0 + 16 * w + 8 * h;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    u[i] = nb + i < a.N ? __ldg(reinterpret_cast<const uint4*>(bank_row(a, l, nb + i) + d0 + 8 * j))
                        : make_uint4(0, 0, 0, 0);
}

// Codes of a loaded tile into W8 (8 bytes per row and thread: a half-warp
// writes one row's 128 contiguous bytes) and, transposed, into W8T.  Each
// thread's 8 x 8 code block is transposed in registers; column col = 8 j + c
// of the tile then holds the thread's 8 codes (rows 16 w + 8 h .. + 7) as one
// 8-byte word, which goes to slot (2 w + h) ^ j of that column's 128-byte
// line in shared memory (the XOR spreads a warp's stores over all banks),
// and the lines leave as 16-byte chunks of W8T rows.
__device__ __forceinline__ void bank_convert_tile(const BankArgs& a, int l, int n0, int d0, const uint4 (&u)[8],
                                                  const Bracket2& kb, uint2 (*trT)[16]) {
  const int w = threadIdx.x >> 5, h = (threadIdx.x >> 4) & 1, j = threadIdx.x & 15;
  const int nb = n0 + 16 * w + 8 * h;
  uint8_t* W8 = a.W8 + static_cast<int64_t>(l) * a.N * a.D;
  uint8_t* W8T = a.W8T + static_cast<int64_t>(l) * a.N * a.D;
  uint32_t lo[8], hi[8];   // codes of row i: columns 0-3, 4-7 of the thread's block
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const f2 v[4] = {f2_from_bf16x2(u[i].x), f2_from_bf16x2(u[i].y), f2_from_bf16x2(u[i].z), f2_from_bf16x2(u[i].w)};
    const uint2 c = quant8(v, kb);
    if (nb + i < a.N) *reinterpret_cast<uint2*>(W8 + static_cast<int64_t>(nb + i) * a.D + d0 + 8 * j) = c;
    lo[i] = c.x;
    hi[i] = c.y;
  }
  uint32_t t0[4], t1[4], t2[4], t3[4];
  transpose4x4(lo[0], lo[1], lo[2], lo[3], t0);   // t0[c]: rows 0-3 of column c
  transpose4x4(lo[4], lo[5], lo[6], lo[7], t1);   // t1[c]: rows 4-7 of column c
  transpose4x4(hi[0], hi[1], hi[2], hi[3], t2);   // t2[c]: rows 0-3 of column 4 + c
  transpose4x4(hi[4], hi[5], hi[6], hi[7], t3);
  const int slot = (2 * w + h) ^ j;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    trT[8 * j + c][slot] = make_uint2(t0[c], t1[c]);
    trT[8 * j + 4 + c][slot] = make_uint2(t2[c], t3[c]);
  }
  __syncthreads();
  // chunk k (slots 2 k, 2 k + 1) of column col lies in the aligned slot pair
  // at (2 k ^ (col / 8)) & ~1, its halves swapped when col / 8 is odd
  const int nvalid = min(128, a.N - n0);   // a multiple of 64
  for (int e = threadIdx.x; e < 128 * 8; e += kBankThreads) {
    const int col = e >> 3, k = e & 7, jj = col >> 3;
    if (16 * k < nvalid) {
      uint4 v = *reinterpret_cast<const uint4*>(&trT[col][(2 * k ^ jj) & ~1]);
      if (jj & 1) v = make_uint4(v.z, v.w, v.x, v.y);
      *reinterpret_cast<uint4*>(W8T + static_cast<int64_t>(d0 + col) * a.N + n0 + 16 * k) = v;
    }
  }
}

// grid: resident blocks (at most one per tile), kBankThreads threads.
__global__ void __launch_bounds__(kBankThreads, 4) bank_refresh_kernel(const __grid_constant__ BankArgs a,
                                                                       BankSync* sy, DevStatus st) {
  __shared__ __align__(16) uint2 trT[128][16];   // [tile column][8-row slot, swizzled]
  __shared__ unsigned int claim[2];
  __shared__ float scale_sh;
  __shared__ float wmax[kBankWarps];
  const int tiles_d = a.D / 128;
  const int tpl = (a.N + 127) / 128 * tiles_d;              // tiles per layer
  const unsigned int U = static_cast<unsigned int>(tpl * a.L);
  const int lane = threadIdx.x & 31;
  // thread 0: the count returned to this block's latest amax item, examined
  // at the start of the block's next item (before any wait) or at the end
  int pend_l = -1;
  unsigned int pend_old = 0;
  if (threadIdx.x == 0) claim[0] = atomicAdd(&sy->next, 1u);
  __syncthreads();
  for (int k = 0;; ++k) {
    const unsigned int item = claim[k & 1];
    if (item >= 2 * U) break;
    // the next claim is in flight while this item runs (items only grow, so
    // an amax item is never held behind a wait); its value is stored at the
    // end of the item, so that no thread waits for it before then
    unsigned int next_item = 0;
    if (threadIdx.x == 0) next_item = atomicAdd(&sy->next, 1u);
    const int tile = static_cast<int>(item < U ? item : item - U);
    const int l = tile / tpl, lt = tile % tpl;
    const int n0 = (lt / tiles_d) * 128, d0 = (lt % tiles_d) * 128;
    uint4 u[8];
    bank_load_tile(a, l, n0, d0, u);
    // with this item's loads in flight, examine the previous amax item's
    // count (it completes a layer at most once per layer; publishing here,
    // before any wait, keeps the publication prompt)
    if (threadIdx.x == 0 && pend_l >= 0) {
      bank_publish_if_last(a, sy, pend_l, pend_old, tpl);
      pend_l = -1;
    }
    if (item < U) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, absmax_bf16x8(u[i]));
      m = warp_max(m);
      if (lane == 0) wmax[threadIdx.x >> 5] = m;
      __syncthreads();
      if (threadIdx.x == 0) {
        float mm = wmax[0];
#pragma unroll
        for (int w = 1; w < kBankWarps; ++w) mm = fmaxf(mm, wmax[w]);
        // the tile's maximum, then the count (released after the maximum)
        red_max_u32(&sy->amax[l], __float_as_uint(mm));
        pend_old = atom_add_acq_rel_u32(&sy->done[l], 1u);
        pend_l = l;
      }
    } else {
      // (the tile's loads are in flight while thread 0 waits for the scale)
      if (threadIdx.x == 0) {
        const int* word = reinterpret_cast<const int*>(&sy->scale[l]);
        int sb = ld_acquire_gpu(word);
        if (sb == 0) {
          const uint64_t t0 = globaltimer_ns();
          while ((sb = ld_acquire_gpu(word)) == 0) {
            __nanosleep(32);
            if (globaltimer_ns() - t0 > st.timeout_ns) {
              record_error(st, QKVP_ERR_TIMEOUT, KID_BANK_QUANT);
              break;
            }
          }
        }
        scale_sh = __int_as_float(sb);   // 0 after a timeout: the tile is skipped
      }
      __syncthreads();
      const float s = scale_sh;
      if (s > 0.f) bank_convert_tile(a, l, n0, d0, u, make_bracket2(s), trT);
    }
    if (threadIdx.x == 0) claim[(k + 1) & 1] = next_item;
    __syncthreads();   // the next claim is visible; `trT` and `scale_sh` are free again
  }
  if (threadIdx.x == 0) {
    if (pend_l >= 0) bank_publish_if_last(a, sy, pend_l, pend_old, tpl);
    __threadfence();
    if (atomicAdd(&sy->exited, 1u) == gridDim.x - 1) {
      // every block is past its last item and its last read of the counters
      for (int l = 0; l < a.L; ++l) {
        sy->amax[l] = 0u;
        sy->done[l] = 0u;
        sy->scale[l] = 0u;
      }
      sy->next = 0u;
      sy->exited = 0u;
      __threadfence();
    }
  }
}

cudaError_t launch_bank_refresh(const BankArgs& a, BankSync* sy, DevStatus st, cudaStream_t s) {
  static std::atomic<int> cache[64];   // per device: resident blocks, written once
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int resident = dev < 64 ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (resident <= 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bank_refresh_kernel, kBankThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    resident = sms * per_sm;
    if (dev < 64) cache[dev].store(resident, std::memory_order_relaxed);
  }
  const int64_t tiles = static_cast<int64_t>((a.N + 127) / 128) * (a.D / 128) * a.L;
  const int grid = static_cast<int>(tiles < resident ? tiles : resident);
  bank_refresh_kernel<<<grid, kBankThreads, 0, s>>>(a, sy, st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// x -> x8 [T, D] codes.  Every block first re-reduces the amax partials of
// x (a few KB from L2), then converts 16 values per thread per step: two
// 16-byte loads, one 16-byte store.  T * D is a multiple of 16 (D % 128 == 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 quant16(uint4 u0, uint4 u1, const Bracket& k) {
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  uint32_t q[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    q[j] = quant4_fast(bf16_lo(w[2 * j]), bf16_hi(w[2 * j]), bf16_lo(w[2 * j + 1]), bf16_hi(w[2 * j + 1]), k);
  return make_uint4(q[0], q[1], q[2], q[3]);
}

__global__ void __launch_bounds__(256) x_quant_kernel(const uint16_t* __restrict__ x, int64_t n16,
                                                      uint8_t* __restrict__ x8, const float* partials, int nparts,
                                                      float* x_scale) {
  __shared__ float red[32];
  const float s = scale_from_amax(block_reduce_partials(partials, nparts, red));
  const Bracket k = make_bracket(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *x_scale = s;
  const uint4* src = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(x8);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + stride < n16; i += 2 * stride) {  // two independent groups in flight
    const uint4 a0 = __ldg(src + 2 * i), a1 = __ldg(src + 2 * i + 1);
    const uint4 b0 = __ldg(src + 2 * (i + stride)), b1 = __ldg(src + 2 * (i + stride) + 1);
    dst[i] = quant16(a0, a1, k);
    dst[i + stride] = quant16(b0, b1, k);
  }
  for (; i < n16; i += stride) dst[i] = quant16(__ldg(src + 2 * i), __ldg(src + 2 * i + 1), k);
}

cudaError_t launch_x_quant(const uint16_t* x, int64_t n, uint8_t* x8, const float* partials, int nparts,
                           float* x_scale, int blocks, cudaStream_t s) {
  x_quant_kernel<<<blocks, 256, 0, s>>>(x, n / 16, x8, partials, nparts, x_scale);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// x amax and x quantise in one launch, separated by a grid barrier.
// ---------------------------------------------------------------------------
// Grid barrier: every block's thread 0 arrives; the last to arrive resets the
// count and advances the generation, the others wait (bounded) for that.
__device__ __forceinline__ void grid_barrier(GridBar* bar, const DevStatus& st, int kid) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const int gen = ld_acquire_gpu(&bar->gen);
    __threadfence();   // this block's writes before its arrival
    if (atomicAdd(&bar->count, 1) == static_cast<int>(gridDim.x) - 1) {
      bar->count = 0;
      __threadfence();
      atomicAdd(&bar->gen, 1);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(&bar->gen) == gen) {
        if (globaltimer_ns() - t0 > st.timeout_ns) {
          record_error(st, QKVP_ERR_TIMEOUT, kid);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

constexpr int kFusedThreads = 512;
// Two blocks per SM at no more than 48 registers a thread, so that a quarter
// of the register file stays free for another kernel's block beside them
// (the bank refresh of the same step: 256 threads x 64 registers).
constexpr int kFusedBlocksPerSm = 2;
constexpr int kFusedMaxRegs = 48;

__global__ void __maxnreg__(kFusedMaxRegs) x_amax_quant_kernel(const uint16_t* __restrict__ x, int64_t n16,
                                                                     uint8_t* __restrict__ x8, float* partials,
                                                                     float* x_scale, GridBar* bar, DevStatus st) {
  __shared__ float red[32];
  const uint4* src = reinterpret_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  // 1: amax over this block's groups of 16 values (four groups in flight)
  float m = 0.f;
  int64_t i = i0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __ldg(src + 2 * (i + j * stride));
      v[2 * j + 1] = __ldg(src + 2 * (i + j * stride) + 1);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, absmax_bf16x8(v[j]));
  }
  for (; i < n16; i += stride)
    m = fmaxf(m, fmaxf(absmax_bf16x8(__ldg(src + 2 * i)), absmax_bf16x8(__ldg(src + 2 * i + 1))));
  m = block_max(m, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
  grid_barrier(bar, st, KID_X_QUANT);
  // 2: the scale from every block's partial, then the codes of the same groups
  float pm = 0.f;   // the other blocks' partials, read from L2
  for (int b = threadIdx.x; b < static_cast<int>(gridDim.x); b += blockDim.x) pm = fmaxf(pm, __ldcg(partials + b));
  const float s = scale_from_amax(block_max(pm, red));
  const Bracket k = make_bracket(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *x_scale = s;
  // in the reverse order of step 1: the groups read last are the likeliest
  // to be in L2 still
  // (last use of the lines: they may go first)
  const uint64_t done = l2_policy_evict_first();
  uint4* dst = reinterpret_cast<uint4*>(x8);
  const int64_t cnt = i0 < n16 ? (n16 - 1 - i0) / stride + 1 : 0;   // this thread's groups
  int64_t c = cnt - 1;
  for (; c >= 1; c -= 2) {
    const int64_t ia = i0 + c * stride, ib = ia - stride;
    const uint4 a0 = ldg_hint(src + 2 * ia, done), a1 = ldg_hint(src + 2 * ia + 1, done);
    const uint4 b0 = ldg_hint(src + 2 * ib, done), b1 = ldg_hint(src + 2 * ib + 1, done);
    dst[ia] = quant16(a0, a1, k);
    dst[ib] = quant16(b0, b1, k);
  }
  if (c == 0) dst[i0] = quant16(ldg_hint(src + 2 * i0, done), ldg_hint(src + 2 * i0 + 1, done), k);
}

cudaError_t launch_x_amax_quant(const uint16_t* x, int64_t n, uint8_t* x8, float* partials, float* x_scale,
                                GridBar* bar, DevStatus st, cudaStream_t s) {
  static std::atomic<int> cache[64];   // per device, written once
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int blocks = dev < 64 ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (blocks <= 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, x_amax_quant_kernel, kFusedThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (per_sm > kFusedBlocksPerSm) per_sm = kFusedBlocksPerSm;
    blocks = sms * per_sm < kMaxFusedBlocks ? sms * per_sm : kMaxFusedBlocks;
    if (dev < 64) cache[dev].store(blocks, std::memory_order_relaxed);
  }
  // no more blocks than groups of 16 values (each block then has work in both steps)
  const int64_t n16 = n / 16;
  const int grid = static_cast<int>(n16 < blocks ? (n16 > 0 ? n16 : 1) : blocks);
  x_amax_quant_kernel<<<grid, kFusedThreads, 0, s>>>(x, n16, x8, partials, x_scale, bar, st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// RoPE table, two rotation pairs per entry:
//   table[(j * max_pos + p) * 4 + {0, 1, 2, 3}]
//     = cos(p w_2j), cos(p w_2j+1), sin(p w_2j), sin(p w_2j+1),
// w_i = base^(-2 i / d_qk), j < d_qk / 4, computed in float64.
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(float* table, int max_pos, int quarter, int d_qk, double base) {
  const int64_t n = static_cast<int64_t>(quarter) * max_pos;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(e / max_pos), p = static_cast<int>(e % max_pos);
    float4 out;
    double sn, cs;
    sincos(static_cast<double>(p) * pow(base, -2.0 * (2 * j) / d_qk), &sn, &cs);
    out.x = static_cast<float>(cs);
    out.z = static_cast<float>(sn);
    sincos(static_cast<double>(p) * pow(base, -2.0 * (2 * j + 1) / d_qk), &sn, &cs);
    out.y = static_cast<float>(cs);
    out.w = static_cast<float>(sn);
    reinterpret_cast<float4*>(table)[e] = out;
  }
}

cudaError_t launch_rope_table(float* table, int max_pos, int d_qk, double base, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(d_qk / 4) * max_pos;
  const int blocks = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  rope_table_kernel<<<blocks, 256, 0, s>>>(table, max_pos, d_qk / 4, d_qk, base);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Self-test of the failure path: wait on a barrier nothing arrives on.
// ---------------------------------------------------------------------------
__global__ void selftest_wait_kernel(DevStatus st) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, st, KID_SELFTEST);
  __syncthreads();
}

cudaError_t launch_selftest_wait(DevStatus st, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(st);
  return cudaGetLastError();
}

}  // namespace qkvp
