// fa_bwd_tiles.cuh -- shared-memory tile geometry and operand helpers of the
// backward kernels (fa_bwd128.cu, fa_bwd64.cu): 128-row tiles as TMA writes them,
// 1-D bulk copies, and the X^T = A B^T product over the head dim.
#pragma once
#include "fa_ptx.cuh"

namespace fa {
namespace bwdt {

constexpr int BT = 128;          // rows of every tile (keys or queries)

// Shared-memory geometry of a 128-row tile of head dim HD as TMA writes it: chunks of
// SPAN columns (64, or all 32 at HD = 32) side by side, each in the 128-byte swizzle
// (64-byte at HD = 32), so that UMMA reads it as a K-major operand (k-steps of 16
// columns) or as an MN-major one (k-steps of 16 rows).
template <int HD>
struct Geo {
  static constexpr int SPAN = HD < 64 ? HD : 64;             // columns per chunk
  static constexpr int NCH = HD / SPAN;                      // chunks per tile
  static constexpr int ROWB = SPAN * 2;                      // bytes per chunk row
  static constexpr int CHUNK = BT * ROWB;                    // bytes per chunk
  static constexpr int KPC = SPAN / 16;                      // K-major k-steps per chunk
  static constexpr uint32_t HI = sdesc_hi(8 * ROWB, ROWB == 128 ? UMMA_SW128 : UMMA_SW64);
  static constexpr int KSTEP_MN = 16 * ROWB;                 // MN-major k-step: 16 rows
  // byte offset of K-major k-step kk
  static constexpr uint32_t koff(int kk) { return (kk / KPC) * CHUNK + (kk % KPC) * 32; }
};

// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// X^T = A B^T over the head dim HD into TMEM columns d_tmem: A and B are 128-row
// K-major tiles (HD/64 chunks of 64 columns each), given by their descriptor low
// words (sdesc_lo with LBO 16).
template <int HD>
__device__ __forceinline__ void issue_ab_t_w(uint32_t d_tmem, uint32_t alo, uint32_t blo,
                                             uint32_t idesc) {
  using G = Geo<HD>;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const uint32_t o = G::koff(kk) >> 4;
    umma_ss_w(d_tmem, alo + o, blo + o, G::HI, idesc, kk > 0);
  }
}

}  // namespace bwdt
}  // namespace fa
