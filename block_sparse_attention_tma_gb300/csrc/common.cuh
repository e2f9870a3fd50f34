// common.cuh - sm_103a building blocks shared by the attention kernels:
// mbarriers with bounded waits, TMA tensor/bulk copies, tcgen05 (UMMA) issue,
// TMEM allocation and loads/stores, shared-memory matrix descriptors.
// Everything is inline PTX; no CUTLASS/CuTe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gbattn.h"

namespace gb {

// ---------------------------------------------------------------------------
// Device-side error word. One per translation unit (no relocatable device
// code); each unit exposes a host function that reads and clears it.
// ---------------------------------------------------------------------------
static __device__ int g_dev_err;

__device__ __forceinline__ void raise_dev_error(int code) { atomicCAS(&g_dev_err, 0, code); }

#define GB_DEFINE_ERROR_READER(name)                                              \
  int name() {                                                                    \
    int v = 0;                                                                    \
    if (cudaMemcpyFromSymbol(&v, gb::g_dev_err, sizeof(int)) != cudaSuccess)      \
      return GBATTN_ERR_CUDA;                                                     \
    int z = 0;                                                                    \
    if (v != 0 && cudaMemcpyToSymbol(gb::g_dev_err, &z, sizeof(int)) != cudaSuccess) \
      return GBATTN_ERR_CUDA;                                                     \
    return v;                                                                     \
  }

// A wait that has not finished after this many nanoseconds gives up. Every
// wait in these kernels normally ends within microseconds. A launch may set
// a shorter limit (its parameter block's wait_ns; 0 = this default).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// The abort flag a CTA's roles share (in shared memory) and the time limit
// of their waits. *w reads or writes the flag.
struct WaitCtl {
  volatile int* flag;
  uint64_t limit_ns;
  __device__ __forceinline__ volatile int& operator*() const { return *flag; }
};
__device__ __forceinline__ WaitCtl wait_ctl(volatile int* flag, uint64_t limit_ns) {
  return WaitCtl{flag, limit_ns ? limit_ns : kWaitLimitNs};
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
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

// The spin of mbar_wait after its first probe failed, out of line: a wait
// site then adds only the probe and a call to the kernel's instruction stream
// (the role loops are long, and their instruction fetch is on the per-tile path).
static __device__ __noinline__ bool mbar_wait_spin(uint32_t a, uint32_t parity, volatile int* flag,
                                                   uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(a, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*flag) return false;
      if (global_ns() - t0 > limit_ns) {
        raise_dev_error(GBATTN_ERR_TIMEOUT);
        *flag = 1;
        return false;
      }
    }
  }
}

// Waits for the phase with the given parity to complete. Gives up (returns
// false, raising GBATTN_ERR_TIMEOUT once) after abort.limit_ns, or as soon as
// the abort flag is set by another role of the same CTA.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try(a, parity)) return true;
  return mbar_wait_spin(a, parity, abort.flag, abort.limit_ns);
}

// Bounded wait used only on the way out of an aborted kernel (the same time
// limit as the kernel's other waits).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_ns();
  while (!mbar_try(a, parity)) {
    if (global_ns() - t0 > w.limit_ns) return;
  }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// TMA row gather: four rows r0..r3 of a 2-D tensor map whose box is one row
// high ((swizzle bytes / 2) elements wide), written to dst as consecutive
// rows. The swizzle follows the shared-memory address, so 32 such gathers
// at dst + 4 * k * row_bytes build the same tile a 128-row tiled load does.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int r0, int r1,
                                            int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}
// Row gather with 16-byte asynchronous copies (cp.async, generic proxy).
// The copying threads' completion is tracked on an mbarrier; the thread that
// waits on it issues fence_async_smem() before the tensor cores read the tile.
//
// Copies one 128-row K-major bf16 tile of D columns into the layout a tiled
// TMA load with an SW-byte swizzle writes: D * 2 / SW slabs of 128 rows x SW
// bytes, the 16-byte chunk c of row r of a slab stored at chunk
// c ^ ((r * SW / 128) % (SW / 16)). Tile row r is row ro[r / 32] of lane
// r % 32 of the row-major [rows, D] matrix src. Each warp instruction copies
// 512 / SW whole slab rows (coalesced global reads).
template <int D, int SW>
__device__ __forceinline__ void gather_tile_async(uint8_t* tile, const __nv_bfloat16* src, const int (&ro)[4],
                                                  int lane) {
  constexpr int CPR = SW / 16;   // 16-byte chunks per slab row
  constexpr int RPI = 32 / CPR;  // slab rows per warp instruction
  constexpr int NSLAB = D * 2 / SW;
  constexpr int SLAB = 128 * SW;
  const int c = lane % CPR, h = lane / CPR;
  // row RPI * i + h: its swizzled chunk depends on i only through i % 2
  uint32_t dl[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int r = RPI * q + h;
    dl[q] = smem_u32(tile) + h * SW + ((c ^ ((r * SW / 128) & (CPR - 1))) << 4);
  }
  const char* sl = reinterpret_cast<const char*>(src) + c * 16;
#pragma unroll
  for (int i = 0; i < 4 * CPR; ++i) {
    // rows 32e .. 32e + 31 are copied by instructions e * CPR .. e * CPR + CPR - 1
    const int row = __shfl_sync(0xffffffffu, ro[i / CPR], (RPI * i + h) & 31);
    const char* g = sl + (size_t)row * (D * 2);
    const uint32_t d = dl[i & 1] + RPI * i * SW;
#pragma unroll
    for (int sb = 0; sb < NSLAB; ++sb)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + sb * SLAB), "l"(g + sb * SW) : "memory");
  }
}
// Arrives on bar once every cp.async this thread has issued so far has landed
// (counts as one of the arrivals the barrier was initialised with).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 1-D bulk copy global -> shared. dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Makes generic-proxy writes to shared memory visible to the async proxy
// (tensor core / TMA reads).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA issue, commit, loads/stores, fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
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

// D(tmem) (+)= A(smem desc) * B(smem desc)
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc)
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive (once) on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor kept as two 32-bit halves. Successive MMA
// k-steps only move the start address (low 14 bits of lo), so an issue loop
// adds a compile-time byte offset >> 4 to lo and reuses hi: no 64-bit
// arithmetic on the issuing thread's critical path.
struct SDesc {
  uint32_t lo, hi;
};
__device__ __forceinline__ SDesc make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  SDesc d;
  d.lo = ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
  d.hi = ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (swz << 29);
  return d;
}
// D(tmem) (+)= A(smem) * B(smem); a/b given as descriptor halves.
__device__ __forceinline__ void mma_ss(uint32_t d, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .b64 ad, bd;\n\t.reg .pred p;\n\t"
      "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n\t}" ::"r"(d),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem).
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint32_t blo, uint32_t bhi, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n\t.reg .b64 bd;\n\t.reg .pred p;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}

// K-major operand tile of 128 rows x K (bf16) in `sw`-byte swizzled slabs of
// 128 rows; step kk (16 elements) starts at slab (kk*16)/(sw/2), byte
// (kk*32) % sw. Returns the descriptor-lo increment (bytes >> 4) of step kk.
__host__ __device__ constexpr uint32_t kmajor_step(int kk, int sw, int slab_bytes) {
  return (uint32_t)((((kk * 16) / (sw / 2)) * slab_bytes + (kk * 32) % sw) >> 4);
}
// MN-major operand: step kk covers 16 K-rows of `sw` bytes each.
__host__ __device__ constexpr uint32_t mnmajor_step(int kk, int sw) { return (uint32_t)((kk * 16 * sw) >> 4); }

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B
// format, 15/16 A/B major (1 = MN-major), [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor. swz: 2 = 128-byte swizzle, 4 = 64-byte,
// 6 = 32-byte. lbo/sbo in bytes. Bits 46-47 hold the descriptor version (1).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= (uint64_t)swz << 61;
  return d;
}
__host__ __device__ constexpr uint32_t swz_code(int swizzle_bytes) {
  return swizzle_bytes == 128 ? 2u : (swizzle_bytes == 64 ? 4u : 6u);
}

// TMEM loads/stores, 32 lanes x 32 bit, 16 or 32 consecutive columns per
// thread. The warp reads the 32-lane quarter selected by (warp id % 4).
#define GB_R16(r, o)                                                                                      \
  "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), "=r"(r[o + 5]),       \
      "=r"(r[o + 6]), "=r"(r[o + 7]), "=r"(r[o + 8]), "=r"(r[o + 9]), "=r"(r[o + 10]), "=r"(r[o + 11]), \
      "=r"(r[o + 12]), "=r"(r[o + 13]), "=r"(r[o + 14]), "=r"(r[o + 15])
#define GB_W16(r, o)                                                                                  \
  "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), "r"(r[o + 4]), "r"(r[o + 5]),         \
      "r"(r[o + 6]), "r"(r[o + 7]), "r"(r[o + 8]), "r"(r[o + 9]), "r"(r[o + 10]), "r"(r[o + 11]), \
      "r"(r[o + 12]), "r"(r[o + 13]), "r"(r[o + 14]), "r"(r[o + 15])
#define GB_P16(r, o)                                                                                      \
  "+r"(r[o + 0]), "+r"(r[o + 1]), "+r"(r[o + 2]), "+r"(r[o + 3]), "+r"(r[o + 4]), "+r"(r[o + 5]),       \
      "+r"(r[o + 6]), "+r"(r[o + 7]), "+r"(r[o + 8]), "+r"(r[o + 9]), "+r"(r[o + 10]), "+r"(r[o + 11]), \
      "+r"(r[o + 12]), "+r"(r[o + 13]), "+r"(r[o + 14]), "+r"(r[o + 15])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : GB_R16(r, 0), GB_R16(r, 16)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : GB_R16(r, 0)
      : "r"(taddr));
}
// Completes outstanding tcgen05.ld of this thread. The "+r" operands tie the
// loaded registers to this point so no use is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld32(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : GB_P16(r, 0), GB_P16(r, 16)::"memory");
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : GB_P16(r, 0)::"memory");
}
// Ties further registers (already covered by an earlier wait) to program order.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile("" : GB_P16(r, 0), GB_P16(r, 16)::"memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      GB_W16(r, 0), GB_W16(r, 16)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16};" ::"r"(taddr),
      GB_W16(r, 0)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// CTA pairs (a cluster of two CTAs on two SMs): the tcgen05 operations of a
// pair use .cta_group::2. One thread of the even CTA issues an MMA with
// M = 256 whose A rows and D rows are split 128 / 128 between the two CTAs
// (each CTA's own shared memory / tensor memory at the same offsets) and
// whose B operand is split N / 2 / N / 2 (CTA r provides columns
// [r N/2, (r+1) N/2) of B at the same shared-memory offset). Every tcgen05
// instruction of such a kernel uses .cta_group::2.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrive (release at cluster scope) on an mbarrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
// Non-blocking probe with acquire at cluster scope (arrivals from the peer CTA).
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for barriers the peer CTA arrives on (cluster-scope acquire).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, const WaitCtl& abort) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_cluster(a, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_cluster(a, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort) return false;
      if (global_ns() - t0 > abort.limit_ns) {
        raise_dev_error(GBATTN_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}
// Whole-cluster execution barrier (every thread of both CTAs).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// Tensor-memory allocation of a CTA pair: one warp of each CTA executes it;
// both CTAs get the same columns.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Pair MMA, D(tmem) (+)= A(smem) * B(smem), descriptors as 32-bit halves.
__device__ __forceinline__ void mma2_ss(uint32_t d, uint32_t alo, uint32_t ahi, uint32_t blo, uint32_t bhi,
                                        uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .b64 ad, bd;\n\t.reg .pred p;\n\t"
      "mov.b64 ad, {%1, %2};\n\tmov.b64 bd, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], ad, bd, %5, p;\n\t}" ::"r"(d),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
// Pair MMA, D(tmem) (+)= A(tmem) * B(smem).
__device__ __forceinline__ void mma2_ts(uint32_t d, uint32_t a_tmem, uint32_t blo, uint32_t bhi, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .b64 bd;\n\t.reg .pred p;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], bd, %4, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in both CTAs of the pair when
// every pair MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)0x3)
      : "memory");
}

// ---------------------------------------------------------------------------
// Small math helpers (hardware instructions, no library code)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed fp32 pairs: one sm_100-family instruction does the work of two
// (d0, d1) = (a0 op b0, a1 op b1); round to nearest even, as the scalar ops.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                     float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void sub2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// bf16x2 of two softmax probabilities (finite, >= 0) on the integer pipe:
// the high half of each bit pattern after adding half a bf16 ulp, i.e. round
// to nearest with ties away from zero. The float-to-bf16x2 conversion
// instruction issues to the same unit as ex2, which the softmax loops keep
// busy. An input that is NaN need not stay NaN (0x7FFFFFFF becomes -0); the
// dK/dV kernel, its user, carries the fp32 value on into dS, so a NaN still
// reaches dK.
__device__ __forceinline__ uint32_t pack_bf16_prob(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo) + 0x8000u, __float_as_uint(hi) + 0x8000u, 0x7632);
}

__device__ __forceinline__ int floor_div(int a, int b) {
  int q = a / b;
  return (a % b != 0 && ((a < 0) != (b < 0))) ? q - 1 : q;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace gb
