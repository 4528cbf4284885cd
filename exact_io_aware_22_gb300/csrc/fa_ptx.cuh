// fa_ptx.cuh -- inline-PTX primitives for sm_103a used by the attention kernels:
// mbarriers with bounded waits, TMA tile loads, TMEM allocation, tcgen05 MMA
// (kind::f16, fp32 accumulation in TMEM), commits, TMEM loads/stores, and the
// UMMA shared-memory / instruction descriptors.
#pragma once
#include <mutex>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fa {

// ---------------------------------------------------------------- status word
// Every spin-wait in the kernels is bounded.  A wait that runs out records
// FA_DEV_TIMEOUT in the status word that the host reads back, and the kernel
// unwinds instead of hanging.
// A kernel that needs every byte of the 227 KiB of shared memory cannot also
// reserve slack to realign it; it checks that the dynamic shared memory starts
// on a 1024-byte boundary (the 128-byte swizzle atom needs it), and if not,
// records FA_DEV_SMEM_ALIGN and returns before touching anything.
enum : uint32_t { FA_DEV_OK = 0u, FA_DEV_TIMEOUT = 1u, FA_DEV_SMEM_ALIGN = 2u };

struct KernelCtl {
  uint32_t* status;         // device status word (sticky OR of FA_DEV_* bits)
  uint64_t wait_limit_ns;   // bound on any single wait
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread for up to `hint_ns` (it resumes as soon as
// the phase completes), so a waiting warp takes no issue slots from the warps
// sharing its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete.  Returns false (and
// records a timeout) if it does not complete within ctl.wait_limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const KernelCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (globaltimer_ns() - t0 > ctl.wait_limit_ns) {
      atomicOr(ctl.status, FA_DEV_TIMEOUT);
      return false;
    }
  }
}

// mbar_wait for code in which every lane of the warp waits and then issues
// warp-wide (.sync.aligned) instructions: the result is the same on all lanes, so
// a lane whose bound ran out never leaves its warp-mates in an aligned
// instruction without it.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const KernelCtl& ctl) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl));
}

// Register split between warpgroups (setmaxnreg): the launch gives every thread the
// kernel's register count; a warpgroup that gives some back (dec) lets another take
// them (inc, which waits until they are free).  Every warp of a warpgroup executes the
// same call.  For a 384-thread CTA launched at 168 registers per thread (64,512 in
// all), one warpgroup at 88 and two at 208 use exactly that total.  Values that live
// across the call must fit the new count, or they go to local memory: with fewer
// than 88, the loaders of the forward and dQ kernels spilled.
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
constexpr uint32_t kRegsLaunch = 168, kRegsLow = 88, kRegsHigh = 208;
static_assert(128 * kRegsLow + 256 * kRegsHigh == 384 * kRegsLaunch,
              "register split must use exactly the launch allocation");
// Host check before launching a kernel that splits its registers: it must have been
// compiled to exactly `launch_regs` registers per thread (kRegsLaunch unless the kernel
// states its own), or the split would not add up (an inc would wait for registers that
// no warpgroup gives back).  Results are kept per kernel; launches from several host
// threads share the record under a lock.
inline cudaError_t check_split_regs(const void* kern, int launch_regs = kRegsLaunch) {
  static std::mutex mu;
  static const void* seen[256];
  static int n_seen = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_seen; ++i)
    if (seen[i] == kern) return cudaSuccess;
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != launch_regs) return cudaErrorInvalidConfiguration;
  if (n_seen < 256) seen[n_seen++] = kern;
  return cudaSuccess;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation (launch_dependent in fa_internal.h) may start while the kernel before
// it in the stream is still running: it sets up (barriers, TMEM) and then waits in
// grid_dep_wait() until that kernel has completed and its writes are visible, before
// touching any global memory that earlier work writes or reads.  grid_dep_launch()
// lets the next kernel in the stream start once every CTA of this grid has called it
// (or exited); it promises nothing about this grid's writes.  Both are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Cluster launch control (dynamic tile scheduling for persistent CTAs).  A running
// CTA asks the hardware to cancel the launch of a CTA that has not started yet and
// takes over its work: try_cancel writes a 16-byte response to shared memory and
// completes 16 transaction bytes on `bar` (the caller has armed it with
// mbar_arrive_expect_tx(bar, 16)); clc_result reads the response and returns the
// x index of the cancelled CTA, or -1 when none was left to cancel.  Once a request
// has come back empty no further request may be made.  The hardware launches (and
// so cancels) CTAs in index order, so a grid ordered longest-first stays so.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp_smem, uint32_t bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
      "[%0], [%1];" ::"r"(resp_smem),
      "r"(bar)
      : "memory");
}
__device__ __forceinline__ int clc_result(uint32_t resp_smem) {
  uint32_t x, ok;
  asm volatile(
      "{\n\t.reg .b128 resp;\n\t.reg .pred p;\n\tld.shared.b128 resp, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, resp;\n\t"
      "selp.u32 %1, 1, 0, p;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, resp;\n\t}"
      : "=r"(x), "=r"(ok)
      : "r"(resp_smem)
      : "memory");
  return ok ? static_cast<int>(x) : -1;
}

// Named barrier among a subset of warps (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 3-D tiled load (x innermost).  x * element size must be a multiple of 16 B.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ---------------------------------------------------------------- TMEM
// Allocation is warp-wide; the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// umma_ss / umma_ts with the shared-memory descriptors given as their words
// (sdesc_lo / sdesc_hi).
__device__ __forceinline__ void umma_ss_w(uint32_t d_tmem, uint32_t alo, uint32_t blo,
                                          uint32_t hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 a, b;\n\tmov.b64 a, {%1, %3};\n\tmov.b64 b, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(alo), "r"(blo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint32_t blo,
                                          uint32_t hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 b;\n\tmov.b64 b, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on an mbarrier when all previously issued tcgen05 async ops of
// this thread have completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Wait for this thread's TMEM loads and tie the loaded registers to the wait,
// so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15]),"+r"(r[16]),"+r"(r[17]),"+r"(r[18]),"+r"(r[19]),"+r"(r[20]),"+r"(r[21]),"+r"(r[22]),"+r"(r[23]),"+r"(r[24]),"+r"(r[25]),"+r"(r[26]),"+r"(r[27]),"+r"(r[28]),"+r"(r[29]),"+r"(r[30]),"+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma operands, TMA stores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors
// Swizzle field of the UMMA shared-memory descriptor (bits 61..63).
enum : uint32_t { UMMA_SW_NONE = 0, UMMA_SW128 = 2, UMMA_SW64 = 4, UMMA_SW32 = 6 };

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (LBO), stride-dimension byte offset (SBO), fixed version field 1 at
// bits 46..47, base offset 0 (tiles are aligned to their swizzle atom), swizzle.
//   K-major, swizzled: rows of one swizzle width along K, 8-row groups SBO apart
//                      (LBO unused while one MMA's K stays inside the row).
//   MN-major, swizzled: one swizzle width along M/N, further M/N chunks LBO
//                      apart; 8-row K groups SBO apart.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swz) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(swz & 7u) << 61;
  return d;
}

// The same descriptor as two 32-bit words.  The high word (SBO, version,
// swizzle) is one constant for all operands of a kernel; the low word (start
// address, LBO) is set up once per buffer, and an offset inside a tile only adds
// offset/16 to it: shared addresses stay below 2^18, so the 14-bit start-address
// field never carries into LBO.
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_hi(uint32_t sbo, uint32_t swz) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | ((swz & 7u) << 29);
}

// Instruction descriptor, kind::f16 with fp32 accumulator: A and B both fp16
// or both bf16; a_mn / b_mn select MN-major operands; N>>3 at bits 17..22,
// M>>4 at bits 24..28.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, bool bf16, bool a_mn,
                                                      bool b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- block order
// Which (batch*head, tile rank) a CTA of a grid of nblk tiles per head takes.
// Heads go in groups of G (8 unless the caller chooses); inside a group every head's
// rank-0 tile comes first, then every head's rank-1 tile, and so on.  Rank 0 is the
// tile with the most work under the causal mask, so the grid runs close to
// longest-first (the short tiles fill the tail), while the CTAs running at one time
// stream the K/V or Q/dO of at most a few heads, which stay in L2.  A G as large as
// the head count orders the whole grid longest-first, which the persistent kernels
// take when every head's streamed tiles fit in L2 together.
struct BlockPos {
  int bh, rank;
};
__device__ __forceinline__ BlockPos block_pos(int nblk, int bid, int G = 8) {
  const int BH = static_cast<int>(gridDim.x) / nblk;
  const int g0 = bid / (G * nblk) * G;
  const int gsz = min(G, BH - g0);
  const int w = bid - g0 * nblk;
  return {g0 + w % gsz, w / gsz};
}
__device__ __forceinline__ BlockPos block_pos(int nblk) {
  return block_pos(nblk, static_cast<int>(blockIdx.x));
}

// ---------------------------------------------------------------- sequence rows
// Where the rows of one attention head live.  Dense (B, H, N, d) tensors have TMA
// maps (d, N, B*H): row r of flat head bh sits at (y, z) = (r, bh).  Packed
// variable-length sequences (total, Hx, d) have maps (d, Hx, total): row r of head
// hx of batch b sits at (hx, first token of b + r), and the sequence has its own
// length.  `head` below is the flat head index for dense tensors and the head within
// the batch for packed ones.
struct SeqRows {
  int base;      // packed: first token of the sequence
  int n;         // rows of the sequence (dense: N)
  bool packed;
  __device__ __forceinline__ int y(int r, int head) const { return packed ? head : r; }
  __device__ __forceinline__ int z(int r, int head) const { return packed ? base + r : head; }
  // element offset of row r of `head` in a tensor of Hx heads of d columns
  __device__ __forceinline__ size_t off(int r, int head, int Hx, int N, int d) const {
    return (packed ? static_cast<size_t>(base + r) * Hx + head
                   : static_cast<size_t>(head) * N + r) * d;
  }
};
// Offsets come from the caller: a sequence is clamped to [0, total) and to N rows
// (the longest sequence), so malformed offsets cannot send a kernel outside the
// tensors -- rows outside are simply not computed.
__device__ __forceinline__ SeqRows seq_rows(const int* __restrict__ cu, int b, int N, int total) {
  if (!cu) return {0, N, false};
  const int a = min(max(__ldg(cu + b), 0), total);
  const int e = min(max(__ldg(cu + b + 1), a), total);
  return {a, min(e - a, N), true};
}
// The same for a kernel instantiated for one layout: PACKED is then a compile-time
// fact, and the dense instantiation carries none of the packed addressing.
template <bool PACKED>
__device__ __forceinline__ SeqRows seq_rows_t(const int* __restrict__ cu, int b, int N, int total) {
  if constexpr (PACKED) {
    const int a = min(max(__ldg(cu + b), 0), total);
    const int e = min(max(__ldg(cu + b + 1), a), total);
    return {a, min(e - a, N), true};
  } else {
    return {0, N, false};
  }
}

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic: two lanes per instruction,
// each rounded exactly like the scalar operation).
__device__ __forceinline__ uint64_t f2_bits(float2 v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 bits_f2(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return bits_f2(d);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of a row of 128 fp32 values held as bits, as a tree of 3-input maxima
// (depth 5), so the 64 max operations do not form a few long dependent chains.
__device__ __forceinline__ float row_max128(const uint32_t (&s)[128]) {
  float a[43], b[15], c[5];
#pragma unroll
  for (int i = 0; i < 42; ++i)
    a[i] = fmax3(__uint_as_float(s[3 * i]), __uint_as_float(s[3 * i + 1]),
                 __uint_as_float(s[3 * i + 2]));
  a[42] = fmaxf(__uint_as_float(s[126]), __uint_as_float(s[127]));
#pragma unroll
  for (int i = 0; i < 14; ++i) b[i] = fmax3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[14] = a[42];
#pragma unroll
  for (int i = 0; i < 5; ++i) c[i] = fmax3(b[3 * i], b[3 * i + 1], b[3 * i + 2]);
  return fmaxf(fmax3(c[0], c[1], c[2]), fmaxf(c[3], c[4]));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
  if constexpr (BF16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  }
}

}  // namespace fa
