// Device helpers shared by the qkvp kernels: inline PTX for mbarriers, TMA
// (cp.async.bulk.tensor), tcgen05 (MMA, TMEM alloc/ld), bounded waits, the
// device status word and the E4M3 / bf16 conversions.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "../../include/qkvp.h"

namespace qkvp {

// Kernel ids recorded beside an error in the status word.
enum KernelId : int {
  KID_BANK_AMAX = 1, KID_BANK_QUANT = 2, KID_X_AMAX = 3, KID_X_QUANT = 4,
  KID_FWD_GEMM = 5, KID_BWD_AMAX = 6, KID_BWD_QUANT = 7, KID_DX_GEMM = 8,
  KID_DW_GEMM = 9, KID_DW_REDUCE = 10, KID_SELFTEST = 11, KID_ROPE = 12
};

struct DevStatus {
  int* word;              // [0] = first error code, [1] = kernel id
  uint64_t timeout_ns;    // limit for every bounded wait
};

__device__ __forceinline__ void record_error(const DevStatus& st, int code, int kid) {
  if (atomicCAS(st.word, 0, code) == 0) atomicExch(st.word + 1, kid);
}

// ---------------------------------------------------------------------------
// Small helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test with acquire semantics at cluster scope (for phases completed
// by arrivals from the other CTA of a pair).
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
template <bool CL>
__device__ __forceinline__ bool mbar_try_wait_t(uint64_t* bar, uint32_t parity) {
  return CL ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity);
}

// Polling part of mbar_wait (below), kept out of line.
template <bool CL = false>
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                   const DevStatus& st, int kid) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait_t<CL>(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > st.timeout_ns) {
      record_error(st, QKVP_ERR_TIMEOUT, kid);
      if (abort != nullptr) *abort = 1;
      return false;
    }
  }
}
// Wait until the phase with parity `parity` of `bar` has completed.  Bounded:
// gives up after st.timeout_ns, or as soon as another role of the CTA has set
// *abort.  On expiry records QKVP_ERR_TIMEOUT and sets *abort.  Returns true
// when the phase completed.  A phase that has already completed costs one
// inline test.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, const DevStatus& st,
                                          int kid) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow<false>(bar, parity, abort, st, kid);
}
// mbar_wait with acquire semantics at cluster scope.
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, volatile int* abort, const DevStatus& st,
                                             int kid) {
  return mbar_try_wait_cl(bar, parity) || mbar_wait_slow<true>(bar, parity, abort, st, kid);
}

// ---------------------------------------------------------------------------
// TMA (tensor) loads and stores, bulk groups, proxy fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// The same load with the completion signalled on the mbarrier at
// shared::cluster address `bar`; with CG2 (cta_group::2) that barrier may sit
// in either CTA of a 2-CTA pair (the destination is this CTA's own memory).
template <bool CG2>
__device__ __forceinline__ void tma_load_2d_at(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  if (CG2)
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// L2 eviction-priority policies for loads that carry a cache hint.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// As tma_load_3d, with an L2 eviction-priority policy for the loaded lines.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                 int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
      "{%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Make generic-proxy writes to shared memory visible to the async proxy (TMA).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 x E4M3 -> F32, one CTA.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// The same operations for a pair of CTAs (a 2-CTA cluster) sharing one MMA
// (cta_group::2): allocation and release are collective (one warp in each
// CTA), the even CTA issues the MMAs (M = 256: A rows 0-127 from its shared
// memory, 128-255 from its peer's at the same offsets; B's N columns split
// in halves the same way; D rows land in each CTA's own TMEM lanes), and
// commits arrive on the barrier at the same offset in both CTAs.  Every
// tcgen05 operation of a kernel uses one CTA-group size, hence the template.
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc_t(uint32_t* dst_smem, uint32_t ncols) {
  if (PAIR)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
  else
    tmem_alloc(dst_smem, ncols);
}
template <bool PAIR>
__device__ __forceinline__ void tmem_relinquish_t() {
  if (PAIR)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    tmem_relinquish();
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc_t(uint32_t taddr, uint32_t ncols) {
  if (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    tmem_dealloc(taddr, ncols);
}
template <bool PAIR>
__device__ __forceinline__ void umma_e4m3_t(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  if (PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    umma_e4m3(d_tmem, adesc, bdesc, idesc, accumulate);
}
// Arrive on `bar` (in both CTAs of the pair for PAIR) once every MMA issued
// so far by this thread has completed.
template <bool PAIR>
__device__ __forceinline__ void umma_commit_t(uint64_t* bar) {
  if (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(static_cast<uint16_t>(3))
        : "memory");
  else
    umma_commit(bar);
}

// ---------------------------------------------------------------------------
// Clusters
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster; release/acquire at cluster scope.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address, in the cluster's shared window, of this CTA's shared variable `p`
// as it sits in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_rank(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrive (release at cluster scope) on an mbarrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Instruction descriptor for kind::f8f6f4: D = F32, A = B = E4M3, both
// K-major, dense, no negation.  Bit fields: [4,6) D format (1 = F32),
// [7,10) A format (0 = E4M3), [10,13) B format, [15] A MN-major, [16] B
// MN-major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for an operand laid out by TMA with
// 128-byte swizzling, general form: [0,14) start address >> 4, [16,30)
// leading byte offset >> 4, [32,46) stride byte offset >> 4, [46,48) version
// 1, [61,64) layout 2 (128-byte swizzle).
//   K-major: rows of 128 bytes of K, 8-row atoms stacked along M/N every
//            `sbo` bytes; the leading offset is unused.
//   MN-major: 128 consecutive M/N elements per 128-byte row, rows along K;
//            8-row atoms stacked along K every `sbo` bytes, 128-element
//            column blocks along M/N every `lbo` bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor as above with A and/or B read MN-major (bit 15 for
// A, bit 16 for B; allowed for 8-bit operands).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32_major(int M, int N, bool a_mn, bool b_mn) {
  return idesc_e4m3_f32(M, N) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u);
}

// Shared-memory matrix descriptor for a K-major operand laid out by TMA with
// 128-byte swizzling: rows of 128 bytes, 8-row (1024 B) swizzle atoms stacked
// along M/N.  Fields: [0,14) start address >> 4, [16,30) leading byte offset
// >> 4 (unused for swizzled K-major), [32,46) stride byte offset >> 4 (1024 B
// between 8-row groups), [46,48) descriptor version (1), [61,64) layout
// (2 = 128-byte swizzle).  The atom base must be 1024-byte aligned; moving
// along K inside the 128-byte row is a plain start-address offset.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp receives
// columns [col, col+16) of TMEM lane (warp's lane-quarter base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Numerics
// ---------------------------------------------------------------------------
// One E4M3FN code (round-to-nearest-even, saturating) of v/s with float32
// IEEE division.
__device__ __forceinline__ uint32_t quant1(float v, float s) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(v, s), __NV_SATFINITE, __NV_E4M3));
}
// Four codes packed little-endian (a in the lowest byte).
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float s) {
  return quant1(a, s) | (quant1(b, s) << 8) | (quant1(c, s) << 16) | (quant1(d, s) << 24);
}

// Exact codes from multiplications.  With rs = fl(1/s), lo = fl(rs (1 - 2^-20))
// and hi = fl(rs (1 + 2^-20)) (a Bracket), fl(v lo) and fl(v hi) lie on either
// side of the IEEE quotient fl(v/s): each product is within 3 * 2^-24 of
// v/s (1 -+ 2^-20) and the quotient within 2^-24 of v/s.  Rounding onto the
// E4M3 grid with saturation is monotone, so when both products give the same
// code that is the quotient's code; otherwise (v/s within ~2^-20 of a
// rounding boundary, rare) the exact division decides.  Products below the
// smallest E4M3 step give a signed zero of v's sign on both sides, as the
// quotient does; |v/s| <= 448 (1 + 2^-23) for the tensors quantised here, so
// no product overflows.
struct Bracket {
  float s, lo, hi;
};
__device__ __forceinline__ Bracket make_bracket(float s) {
  const float rs = __frcp_rn(s);
  return Bracket{s, rs * 0.99999904632568359375f, rs * 1.00000095367431640625f};
}

// The rare exact path, kept out of line so the division is executed only when
// a bracket straddles a rounding boundary (not predicated for every value).
static __device__ __noinline__ uint32_t quant2_exact(float a, float b, float s) {
  return quant1(a, s) | (quant1(b, s) << 8);
}

// Two codes (a in the low byte).
__device__ __forceinline__ uint32_t quant2_fast(float a, float b, const Bracket& k) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a * k.lo, b * k.lo), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(a * k.hi, b * k.hi), __NV_SATFINITE, __NV_E4M3);
  if (__builtin_expect(lo == hi, 1)) {
    // __nv_cvt_float2_to_fp8x2 puts .x in the low byte
    return lo;
  }
  return quant2_exact(a, b, k.s);
}
// Four codes packed little-endian (a in the lowest byte).
__device__ __forceinline__ uint32_t quant4_fast(float a, float b, float c, float d, const Bracket& k) {
  return quant2_fast(a, b, k) | (quant2_fast(c, d, k) << 16);
}

// ---------------------------------------------------------------------------
// Packed float32 pairs: two lanes of one 64-bit register, for the f32x2
// arithmetic of sm_100 and later (each lane rounds exactly as the scalar
// instruction does).
// ---------------------------------------------------------------------------
using f2 = uint64_t;
__device__ __forceinline__ f2 f2_make(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_split(f2 a) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(a));
  return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// a * b + c, one rounding per lane
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// The two bf16 of a word (low half first) as a float pair, exactly.
__device__ __forceinline__ f2 f2_from_bf16x2(uint32_t w) {
  return f2_make(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// Both lanes rounded to bf16 and packed (lane 0 in the low half).
__device__ __forceinline__ uint32_t f2_to_bf16x2(f2 a) {
  const float2 v = f2_split(a);
  __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<uint32_t*>(&h);
}
// max(a, b, c) (three-operand form of sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// Running max of |lane| over a pair.
__device__ __forceinline__ float f2_absmax(float m, f2 a) {
  const float2 v = f2_split(a);
  return fmax3(m, fabsf(v.x), fabsf(v.y));
}

// Eight codes (little-endian, lane 0 of v[0] lowest) with the bracket test
// made once for all eight; the exact division is taken only when a bracket
// straddles a rounding boundary.
static __device__ __noinline__ uint2 quant8_exact(f2 v0, f2 v1, f2 v2, f2 v3, float s) {
  const float2 a = f2_split(v0), b = f2_split(v1), c = f2_split(v2), d = f2_split(v3);
  return make_uint2(quant1(a.x, s) | (quant1(a.y, s) << 8) | (quant1(b.x, s) << 16) | (quant1(b.y, s) << 24),
                    quant1(c.x, s) | (quant1(c.y, s) << 8) | (quant1(d.x, s) << 16) | (quant1(d.y, s) << 24));
}
struct Bracket2 {
  float s;
  f2 lo, hi;   // both lanes rs(1 - 2^-20), rs(1 + 2^-20)
};
__device__ __forceinline__ Bracket2 make_bracket2(float s) {
  const Bracket k = make_bracket(s);
  return Bracket2{s, f2_make(k.lo, k.lo), f2_make(k.hi, k.hi)};
}
__device__ __forceinline__ uint32_t cvt_e4m3x2(f2 a) {
  const float2 v = f2_split(a);
  return __nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3);   // .x in the low byte
}
__device__ __forceinline__ uint2 quant8(const f2 (&v)[4], const Bracket2& k) {
  const uint32_t l0 = cvt_e4m3x2(f2_mul(v[0], k.lo)) | (cvt_e4m3x2(f2_mul(v[1], k.lo)) << 16);
  const uint32_t l1 = cvt_e4m3x2(f2_mul(v[2], k.lo)) | (cvt_e4m3x2(f2_mul(v[3], k.lo)) << 16);
  const uint32_t h0 = cvt_e4m3x2(f2_mul(v[0], k.hi)) | (cvt_e4m3x2(f2_mul(v[1], k.hi)) << 16);
  const uint32_t h1 = cvt_e4m3x2(f2_mul(v[2], k.hi)) | (cvt_e4m3x2(f2_mul(v[3], k.hi)) << 16);
  if (__builtin_expect(((l0 ^ h0) | (l1 ^ h1)) == 0, 1)) return make_uint2(l0, l1);
  return quant8_exact(v[0], v[1], v[2], v[3], k.s);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Scale from an amax: amax / 448 in float32, 1 when amax == 0.
__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide max of one value per thread; result valid in every thread.
// red_smem: >= 32 floats.  Every thread of the block must call it.
__device__ __forceinline__ float block_max(float v, float* red_smem) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  if ((threadIdx.x & 31) == 0) red_smem[w] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float x = threadIdx.x < nw ? red_smem[threadIdx.x] : 0.f;
    x = warp_max(x);
    if (threadIdx.x == 0) red_smem[0] = x;
  }
  __syncthreads();
  const float r = red_smem[0];
  __syncthreads();
  return r;
}

// Max over `n` partial maxima (non-negative floats) by one block.
__device__ __forceinline__ float block_reduce_partials(const float* partials, int n, float* red_smem) {
  float m = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, partials[i]);
  return block_max(m, red_smem);
}

}  // namespace qkvp
