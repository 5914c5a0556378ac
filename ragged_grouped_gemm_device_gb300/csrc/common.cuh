// Device helpers shared by the kernels: inline PTX for mbarriers, TMA (cp.async.bulk.tensor),
// tcgen05 (tensor-memory allocation, MMA, commit, loads) and bounded waits.
//
// Every wait in this library is bounded: after `timeout_ns` of %globaltimer time a waiting thread
// records MOE_DEV_TIMEOUT in the caller's status word, raises the CTA's abort flag and returns
// false, so that a lost arrival turns into an error status rather than a hung GPU.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/moe_gg.h"
#include "debug.cuh"

namespace moe {

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_status(int32_t* status, int bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// `count` arrivals at once.
__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase of parity `parity` of barrier `bar` has completed. Gives up (returns
// false) when the CTA's abort flag is raised, or after timeout_ns, in which case it raises the
// flag and records MOE_DEV_TIMEOUT. `honour_abort` = false is used by teardown waits that must
// drain in-flight copies even after an abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status, long long timeout_ns,
                                          bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  // try_wait itself suspends the thread for a while when the phase is not complete, so the
  // clock and the abort flag are checked after every unsuccessful try
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *abort_flag) return false;
    if (static_cast<long long>(globaltimer_ns() - t0) > timeout_ns) {
      *abort_flag = 1;
      record_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// The shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address, which may lie in another CTA of
// the cluster (default release semantics; see the pair protocol in the grouped GEMM kernel for
// what each such arrival orders).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Every thread of every CTA of the cluster arrives, then waits for all of them.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// As tma_load_2d for the odd CTA of a pair (tcgen05 cta_group::2 kernels): the box lands in this
// CTA's shared memory at `dst` and its bytes complete on the mbarrier at the shared::cluster
// address `cluster_bar`, which may be the even CTA's.
__device__ __forceinline__ void tma_load_2d_peer(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cluster_bar)
      : "memory");
}

// Untiled bulk copy global -> shared of `bytes` (a multiple of 16; both addresses 16-byte
// aligned), completing on the mbarrier `bar` like the tensor loads.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Shared -> global tensor store (clipped at the tensor's bounds), tracked by a bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until the shared-memory source of every committed bulk store has been read.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ... all but the most recently committed one.
__device__ __forceinline__ void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy writes to shared memory made visible to the async proxy (tensor core reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ... for writes to the shared memory of any CTA of the cluster.
__device__ __forceinline__ void fence_proxy_async_cluster() {
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}

// 16 zero bytes at a shared::cluster address (possibly another CTA's shared memory).
__device__ __forceinline__ void st_cluster_zero16(uint32_t cluster_addr) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(cluster_addr), "r"(0u) : "memory");
}

// ---------------------------------------------------------------------------------- tcgen05
// The allocation instructions take the CTA group of the kernel's MMAs (every tcgen05
// instruction of a kernel names the same group). With CG = 2 one warp of each CTA of the pair
// executes them together and both CTAs get the same columns.
template <int CG = 1>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

template <int CG = 1>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (CG == 2)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int CG = 1>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 inputs, fp32 accumulator).
// With CG = 2 (issued by the even CTA of a pair) the MMA is M = 256 rows over the two CTAs:
// each CTA's shared memory holds its 128 rows of A and half of B's N rows at the descriptors'
// offsets, and each CTA's tensor memory receives its 128 rows of D at d_tmem.
template <int CG = 1>
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  if constexpr (CG == 2)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed. `bar`
// is a shared::cluster address: with CG = 2 it may be the peer CTA's barrier.
template <int CG = 1>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  if constexpr (CG == 2)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Block-scaled D[tmem] (+)= (A * SA) * (B * SB)^T, kind::mxf8f6f4 with one E8M0 scale per 32
// elements of K (scale_vec::1X): A and B from shared-memory descriptors, the scales of A's
// rows and B's rows from tensor memory at sfa / sfb; the instruction descriptor's scale ids
// pick the byte of each 32-bit scale word (the K-step within a 4-step chunk).
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared -> tensor memory copy of 32 rows x 128 bits, replicated into the four lane quadrants:
// row i of the source lands in lane i of every quadrant, 4 consecutive columns from `taddr`.
// Ordered before the tcgen05.mma instructions this thread issues after it.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 32 lanes x 16 columns of 32-bit words: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Wait for this thread's tcgen05.ld results; the registers are threaded through the asm so
// the compiler cannot hoist their uses above the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld_wait2(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                 "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                 "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(b[0]), "+r"(b[1]),
                 "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
                 "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
                 "+r"(b[14]), "+r"(b[15])
               :
               : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes from registers (lane i of the warp
// writes lane i of its quadrant), and the wait for this thread's outstanding tcgen05.st.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and stride byte
// offsets (16-byte units), descriptor version 1 at bit 46, 128-byte swizzle (mode 2) at bit 61.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Shared-memory descriptor of an unswizzled region of 16-byte rows stored back to back (the
// 8-row core matrices 128 bytes apart in both directions), for tcgen05.cp.
__device__ __forceinline__ uint64_t smem_desc_rows16(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
         (static_cast<uint64_t>(128 >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor for kind::mxf8f6f4 with block scaling: E4M3 A and B (format 0), both
// K-major, fp32 accumulator (implied), E8M0 scales (bit 23), N, M; the scale-id fields (bits
// 29-30 for A, 4-5 for B) are or-ed in per K-step.
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(int M, int N) {
  return ((static_cast<uint32_t>(N) >> 3) << 17) | (1u << 23) | ((static_cast<uint32_t>(M) >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_sf_ids(uint32_t ks) { return (ks << 29) | (ks << 4); }

// Instruction descriptor for kind::f16: fp32 accumulator, bf16 A and B, operand majors, N, M.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

// ---------------------------------------------------------------------------------- MXFP8
// OCP MXFP8 element and scale encoding, shared by every kernel that quantizes (so that the
// codes agree bit for bit whichever kernel produced them).
// Shared exponent of a block from its largest magnitude (fp32, exact for bf16 inputs).
__device__ __forceinline__ int mx_exponent(float amax) {
  const int eb = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  if (eb == 0) return -127;               // zero or subnormal max: floor(log2) - 8 < -127
  return max(eb - 127 - 8, -127);         // normal: floor(log2(amax)) = eb - 127
}

// 1 / 2^s for s in [-127, 126]: a normal fp32 power of two
__device__ __forceinline__ float mx_inv_scale(int s) { return __uint_as_float(static_cast<uint32_t>(127 - s) << 23); }

// a in the low byte, b in the high byte (memory order of two consecutive elements)
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  const uint32_t ca = __nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3);
  const uint32_t cb = __nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3);
  return (ca & 0xFFu) | ((cb & 0xFFu) << 8);
}

// Byte of the scale of row r (0..127 of its 128-row tile G) and 32-block kb (counted from the
// row's start) in the atoms of an operand with KC 128-element chunks per row.
__device__ __forceinline__ size_t atom_byte(long long G, int KC, int kb_global, int r) {
  return static_cast<size_t>(G * KC + (kb_global >> 2)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (kb_global & 3);
}

// ---------------------------------------------------------------------------------- bf16 packing
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// One MXFP8 block of 32 bf16 values given as 16 packed pairs (elements 0..15 in p0, 16..31 in
// p1, lower element of a pair in the low half): 32 E4M3 codes in memory order and the E8M0
// scale code. The same arithmetic as every other quantizer of the library.
__device__ __forceinline__ uint8_t mx_block_bf16(const uint32_t (&p0)[8], const uint32_t (&p1)[8],
                                                 uint32_t (&codes)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(p0[j])), fabsf(bf16_hi(p0[j]))));
    amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(p1[j])), fabsf(bf16_hi(p1[j]))));
  }
  const int s = mx_exponent(amax);
  const float inv = mx_inv_scale(s);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    codes[j] = e4m3x2(bf16_lo(p0[2 * j]) * inv, bf16_hi(p0[2 * j]) * inv) |
               (e4m3x2(bf16_lo(p0[2 * j + 1]) * inv, bf16_hi(p0[2 * j + 1]) * inv) << 16);
    codes[4 + j] = e4m3x2(bf16_lo(p1[2 * j]) * inv, bf16_hi(p1[2 * j]) * inv) |
                   (e4m3x2(bf16_lo(p1[2 * j + 1]) * inv, bf16_hi(p1[2 * j + 1]) * inv) << 16);
  }
  return static_cast<uint8_t>(s + 127);
}

}  // namespace moe
