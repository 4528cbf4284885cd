// fa_bwd128.cu -- attention backward (dK/dV and dQ) on sm_103a at head dim 128
// (the pre-pass is in fa_bwd.cu, the persistent kernels for head dims 32 and 64
// in fa_bwd64.cu).  The kernels are templated on HD but instantiated at 128 only.
//
// Method: "flash-attn-triton" docs page, section "Scope" (backward kernels for
// dQ, dK, dV that rebuild P from the saved L; causal mask only on diagonal
// tiles; ragged N) and "Source" (delta pre-pass, then dK/dV, then dQ).
// Gradients follow the chain rule of the forward:
//   P = exp(S - L),  dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),
//   dS = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Two kernels after the pre-pass, both with every tensor product a tcgen05 MMA
// of M = 128, N = 128 (an M = 128 MMA costs about as much at N = 64 as at
// N = 128 on this part, so narrower tiles waste half the tensor rate):
//
//   dkdv_kernel  key-stationary: one CTA per 128-key block, K and V in shared
//                memory, loop over 128-query tiles (causal: from the diagonal
//                down).  TMEM: dV | dK | S^T | dP^T, 128 columns each (dV and dK
//                use HD of theirs).  Once a
//                compute thread holds its 64 dP^T values it writes P^T and then
//                dS^T as 16-bit pairs over those columns, 32 each: the A
//                operands of dV += P^T dO and dK += dS^T Q, so no score tile
//                passes through shared memory, which holds a three-stage Q ring
//                and a two-stage dO ring instead.  The next S^T is issued as soon
//                as the compute warps hold this one; dV starts once P^T is
//                stored, before dS^T is.  Pipe order per tile i: S^T(i+1), dV(i),
//                dK(i), dP^T(i+1).
//   dq_kernel    query-stationary: one CTA per 128-query tile, loop over 128-key
//                blocks (causal: up to the diagonal).  Each compute thread of the
//                first warpgroup copies its row of Q into TMEM once, so S = Q K^T
//                takes its A operand from TMEM; shared memory holds dO and a
//                three-stage K/V ring (one block's loads take longer than its
//                MMAs; two stages left the tensor pipe waiting).  TMEM:
//                dQ | S | dP | Z (64) | Q (HD/2).  S and dP have columns of their
//                own, so the next block's S and dP start as soon as the compute
//                warps hold this block's; dS = P o (dP - D) goes as 16-bit pairs
//                into Z and feeds dQ += dS K from TMEM.
// Recomputing S and dP for dQ costs two extra products, but it needs no
// cross-CTA reduction: accumulating dQ partials in fp32 at L2 from the
// key-stationary kernel is bound by L2 reduction throughput on this part
// (about 3 TB/s, i.e. ~1.4 ms for the 4.4 GB of partials at N = 8192 causal),
// and the split form is deterministic.
//
// Roles in both kernels (384 threads, one CTA per SM):
//   warp 0       TMA producer.   warp 1  TMEM allocator; lane 0 issues MMAs
//                (in dq: S and dP; lane 0 of warp 2 issues dQ).
//   warps 4-11   two compute warpgroups, one thread per TMEM lane (a key row
//                in dkdv, a query row in dq), 64 columns each; in the epilogue
//                warpgroup h stores head-dim columns [64h, 64h + 64).
#include "fa_bwd_tiles.cuh"
#include "fa_internal.h"
#include "fa_ptx.cuh"

#include <type_traits>

namespace fa {

namespace {

using bwdt::BT;
using bwdt::Geo;
using bwdt::bulk_load;
using bwdt::issue_ab_t_w;
constexpr int THREADS = 384;

// Epilogue: NC (32 or 64) fp32 TMEM columns of this thread's lane, times mul,
// rounded to the 16-bit type and stored as one contiguous run of 2 NC bytes (when
// valid).
template <int NC, bool BF16>
__device__ __forceinline__ void store_row(uint32_t taddr, float mul, void* dst, bool valid) {
#pragma unroll
  for (int cc = 0; cc < NC / 16; ++cc) {
    uint32_t v[16];
    tmem_ld16(taddr + 16 * cc, v);
    tmem_ld_wait_regs(v);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
    if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(static_cast<uint8_t*>(dst) + 32 * cc);
      d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

// ============================================================== dK / dV
namespace kv {
// shared memory of head dim HD: K, V resident; Q with L*log2e in a 3-stage ring, dO
// with D in a 2-stage ring; barriers kv_full, q_full[3], q_empty[3], do_full[2],
// do_empty[2], s_full, s_free, dp_full, p_ready, ds_ready, out_full, done
template <int HD>
struct Smem {
  static constexpr int TILE = BT * HD * 2;
  static constexpr int Q_STAGES = 3, DO_STAGES = 2;
  static constexpr int K_OFF = 0, V_OFF = TILE, Q_OFF = 2 * TILE;
  static constexpr int DO_OFF = Q_OFF + Q_STAGES * TILE;
  static constexpr int L_OFF = DO_OFF + DO_STAGES * TILE;   // per Q stage: 128 L*log2e
  static constexpr int D_OFF = L_OFF + Q_STAGES * 512;      // per dO stage: 128 D
  static constexpr int BAR_OFF = D_OFF + DO_STAGES * 512;
  static constexpr int NBARS = 1 + 2 * Q_STAGES + 2 * DO_STAGES + 7;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SMEM_BYTES = SLOT_OFF + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");
};
// dV | dK | S^T | dP^T (dV and dK use their first HD columns).  Once a compute thread holds its 64 dP^T values it writes
// P^T (16-bit pairs) over the first 32 of those columns and dS^T over the last 32.
constexpr uint32_t DV_COL = 0, DK_COL = 128, S_COL = 256, DP_COL = 384;
}  // namespace kv

template <int HD, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    dkdv128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const float* __restrict__ Dp, const float* __restrict__ Lp,
                   void* __restrict__ dK, void* __restrict__ dV, int N, int Np, int group,
                   int window, const int* __restrict__ cu_seqlens, int H, int total, float scale,
                   float c_log2, KernelCtl ctl) {
  using namespace kv;
  using SM = Smem<HD>;
  using G = Geo<HD>;
  constexpr int TILE = SM::TILE, Q_STAGES = SM::Q_STAGES, DO_STAGES = SM::DO_STAGES;
  constexpr int K_OFF = SM::K_OFF, V_OFF = SM::V_OFF, Q_OFF = SM::Q_OFF, DO_OFF = SM::DO_OFF;
  constexpr int L_OFF = SM::L_OFF, D_OFF = SM::D_OFF, BAR_OFF = SM::BAR_OFF, NBARS = SM::NBARS;
  constexpr int SLOT_OFF = SM::SLOT_OFF;
  extern __shared__ __align__(1024) uint8_t sg[];
  const uint32_t sb = smem_u32(sg);
  grid_dep_launch();
  if (sb & 1023u) {                                // see FA_DEV_SMEM_ALIGN
    grid_dep_wait();
    if (threadIdx.x == 0) atomicOr(ctl.status, FA_DEV_SMEM_ALIGN);
    return;
  }
  if (cu_seqlens) grid_dep_wait();                 // the offsets may come from earlier work
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (N + BT - 1) / BT;
  const BlockPos bp = block_pos(nkb);
  const int bkv = bp.bh;                           // K/V head; its query heads: bkv*group + g
  const int kb = bp.rank;                          // causal: block 0 has the most work
  const int q_start = CAUSAL ? kb : 0;             // the diagonal query tile
  const int Hkv = H / group;
  const SeqRows sr = seq_rows(cu_seqlens, bkv / Hkv, N, total);
  const int hk = sr.packed ? bkv % Hkv : bkv;      // K/V head coordinate
  const int nq_r = (sr.n + BT - 1) / BT;           // query tiles of this sequence
  // query tiles per query head: from the diagonal to the last tile that sees a key of
  // this block (with a window of W keys, query rows up to the block's last key + W - 1)
  const int n_head = kb * BT >= sr.n ? 0
      : ((CAUSAL && window > 0) ? min(nq_r, (kb * BT + BT - 1 + window - 1) / BT + 1) : nq_r) -
            q_start;
  const int n_iter = group * n_head;               // the group's query heads one after another
  if (n_iter <= 0) return;                         // a key block past the end of its packed sequence

  auto bar = [&](int i) -> uint32_t { return sb + BAR_OFF + 8 * i; };
  const int B_KV = 0;
  auto B_QF = [&](int s) { return 1 + s; };
  auto B_QE = [&](int s) { return 1 + Q_STAGES + s; };
  auto B_GF = [&](int g) { return 1 + 2 * Q_STAGES + g; };   // dO and D of a stage
  auto B_GE = [&](int g) { return 1 + 2 * Q_STAGES + DO_STAGES + g; };
  const int B_SF = 1 + 2 * Q_STAGES + 2 * DO_STAGES, B_SFREE = B_SF + 1, B_DPF = B_SF + 2,
            B_PR = B_SF + 3, B_DR = B_SF + 4, B_OF = B_SF + 5, B_DONE = B_SF + 6;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_SFREE), 256);
    mbar_init(bar(B_PR), 256);
    mbar_init(bar(B_DR), 256);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SLOT_OFF, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + SLOT_OFF);
  grid_dep_wait();                                 // D and L*log2e from the pre-pass

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_iter > 0) {
      mbar_arrive_expect_tx(bar(B_KV), 2 * TILE);
      for (int c = 0; c < G::NCH; ++c) {
        tma_load_3d(sb + K_OFF + c * G::CHUNK, &tmK, bar(B_KV), c * G::SPAN, sr.y(kb * BT, hk),
                    sr.z(kb * BT, hk));
        tma_load_3d(sb + V_OFF + c * G::CHUNK, &tmV, bar(B_KV), c * G::SPAN, sr.y(kb * BT, hk),
                    sr.z(kb * BT, hk));
      }
      // Q with L*log2e in a three-stage ring, dO with D in a two-stage ring (L and D:
      // padded per-row arrays, 512-byte aligned per tile).  Both stages of a tile are
      // freed by its dK MMAs, the last reader of either.
      bool ok = true;
      int nq_issued = 0, ng_issued = 0;
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % Q_STAGES, g = it % DO_STAGES;
        const int gh = it / n_head;                // which query head of the group
        const int qrow = (q_start + it - gh * n_head) * BT, bhq = bkv * group + gh;
        const int hq = sr.packed ? bhq % H : bhq;
        const size_t row = static_cast<size_t>(bhq) * Np + qrow;
        if (!(ok = mbar_wait(bar(B_QE(s)), ((it / Q_STAGES) & 1) ^ 1, ctl))) break;
        mbar_arrive_expect_tx(bar(B_QF(s)), TILE + 512);
        for (int c = 0; c < G::NCH; ++c)
          tma_load_3d(sb + Q_OFF + s * TILE + c * G::CHUNK, &tmQ, bar(B_QF(s)), c * G::SPAN,
                      sr.y(qrow, hq), sr.z(qrow, hq));
        bulk_load(sb + L_OFF + s * 512, Lp + row, 512, bar(B_QF(s)));
        ++nq_issued;
        if (!(ok = mbar_wait(bar(B_GE(g)), ((it / DO_STAGES) & 1) ^ 1, ctl))) break;
        mbar_arrive_expect_tx(bar(B_GF(g)), TILE + 512);
        for (int c = 0; c < G::NCH; ++c)
          tma_load_3d(sb + DO_OFF + g * TILE + c * G::CHUNK, &tmdO, bar(B_GF(g)), c * G::SPAN,
                      sr.y(qrow, hq), sr.z(qrow, hq));
        bulk_load(sb + D_OFF + g * 512, Dp + row, 512, bar(B_GF(g)));
        ++ng_issued;
      }
      if (!ok) {
        mbar_wait(bar(B_KV), 0, ctl);
        for (int jj = max(0, nq_issued - Q_STAGES); jj < nq_issued; ++jj)
          mbar_wait(bar(B_QF(jj % Q_STAGES)), (jj / Q_STAGES) & 1, ctl);
        for (int jj = max(0, ng_issued - DO_STAGES); jj < ng_issued; ++jj)
          mbar_wait(bar(B_GF(jj % DO_STAGES)), (jj / DO_STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = umma_idesc_f16(BT, BT, BF16, false, false);   // S^T, dP^T
      constexpr uint32_t idG = umma_idesc_f16(BT, HD, BF16, false, true);    // dV, dK
      // descriptor low words: K, V and stage 0 of the Q and dO rings, K-major (LBO 16,
      // for S^T and dP^T) and MN-major (LBO = one 64-column chunk, for dK and dV); a
      // stage is TILE bytes on
      constexpr uint32_t HI = G::HI, STAGE_W = TILE >> 4;
      const uint32_t k_lo = sdesc_lo(sb + K_OFF, 16), v_lo = sdesc_lo(sb + V_OFF, 16);
      const uint32_t q_lo = sdesc_lo(sb + Q_OFF, 16), qm_lo = sdesc_lo(sb + Q_OFF, G::CHUNK);
      const uint32_t o_lo = sdesc_lo(sb + DO_OFF, 16), om_lo = sdesc_lo(sb + DO_OFF, G::CHUNK);
      bool ok = mbar_wait(bar(B_KV), 0, ctl) && mbar_wait(bar(B_QF(0)), 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_ab_t_w<HD>(tmem + S_COL, k_lo, q_lo, idS);
        umma_commit(bar(B_SF));
        if ((ok = mbar_wait(bar(B_GF(0)), 0, ctl))) {
          tc_fence_after();
          issue_ab_t_w<HD>(tmem + DP_COL, v_lo, o_lo, idS);
          umma_commit(bar(B_DPF));
        }
      }
      for (int it = 0; ok && it < n_iter; ++it) {
        const int s = it % Q_STAGES, g = it % DO_STAGES;
        const bool next = it + 1 < n_iter;
        if (next) {
          // the next S^T as soon as the compute warps hold this one
          const int s1 = (it + 1) % Q_STAGES;
          if (!(ok = mbar_wait(bar(B_QF(s1)), ((it + 1) / Q_STAGES) & 1, ctl))) break;
          if (!(ok = mbar_wait(bar(B_SFREE), it & 1, ctl))) break;
          tc_fence_after();
          issue_ab_t_w<HD>(tmem + S_COL, k_lo, q_lo + s1 * STAGE_W, idS);
          umma_commit(bar(B_SF));
        }
        // dV += P^T dO, P^T from the first half of each warpgroup's dP^T columns
        if (!(ok = mbar_wait(bar(B_PR), it & 1, ctl))) break;
        tc_fence_after();
        const uint32_t dv_b = om_lo + g * STAGE_W, acc0 = it > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          umma_ts_w(tmem + DV_COL, tmem + DP_COL + (kk / 4) * 64 + (kk % 4) * 8,
                    dv_b + kk * (G::KSTEP_MN >> 4), HI, idG, kk > 0 ? 1u : acc0);
        // dK += dS^T Q, dS^T from the second half
        if (!(ok = mbar_wait(bar(B_DR), it & 1, ctl))) break;
        tc_fence_after();
        const uint32_t dk_b = qm_lo + s * STAGE_W;
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          umma_ts_w(tmem + DK_COL, tmem + DP_COL + (kk / 4) * 64 + 32 + (kk % 4) * 8,
                    dk_b + kk * (G::KSTEP_MN >> 4), HI, idG, kk > 0 ? 1u : acc0);
        umma_commit(bar(B_QE(s)));
        umma_commit(bar(B_GE(g)));
        if (next) {
          // the next dP^T over P^T and dS^T: issued after the MMAs that read them
          const int g1 = (it + 1) % DO_STAGES;
          if (!(ok = mbar_wait(bar(B_GF(g1)), ((it + 1) / DO_STAGES) & 1, ctl))) break;
          tc_fence_after();
          issue_ab_t_w<HD>(tmem + DP_COL, v_lo, o_lo + g1 * STAGE_W, idS);
          umma_commit(bar(B_DPF));
        }
      }
      if (ok) umma_commit(bar(B_OF));
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ compute
    const int h = (warp - 4) >> 2;                 // query columns [64h, 64h + 64)
    const int kr = (warp & 3) * 32 + lane;         // key row (= TMEM lane)
    const int gkey = kb * BT + kr;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + S_COL + 64 * h;
    const uint32_t tP = tmem + lane_off + DP_COL + 64 * h;
    const float2 c2 = make_float2(c_log2, c_log2);
    bool ok = n_iter > 0;
    for (int it = 0, itl = 0; ok && it < n_iter; ++it, itl = itl + 1 == n_head ? 0 : itl + 1) {
      const int s = it % Q_STAGES, g = it % DO_STAGES;
      if (!(ok = mbar_wait_warp(bar(B_SF), it & 1, ctl))) break;
      tc_fence_after();
      uint32_t x[64];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tc_fence_before();
      mbar_arrive(bar(B_SFREE));                   // S^T may now receive the next tile
      if (!(ok = mbar_wait_warp(bar(B_QF(s)), (it / Q_STAGES) & 1, ctl))) break;
      const float* Ls = reinterpret_cast<const float*>(sg + L_OFF + s * 512) + 64 * h;
      // P^T = exp2(S^T c - L log2e); on the diagonal tile, zero where the query precedes
      // the key
      float p[64];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = *reinterpret_cast<const float4*>(Ls + 4 * c4);
        const float2 t0 = fma2(make_float2(__uint_as_float(x[4 * c4]), __uint_as_float(x[4 * c4 + 1])),
                               c2, make_float2(-l4.x, -l4.y));
        const float2 t1 = fma2(make_float2(__uint_as_float(x[4 * c4 + 2]), __uint_as_float(x[4 * c4 + 3])),
                               c2, make_float2(-l4.z, -l4.w));
        p[4 * c4] = ex2(t0.x);
        p[4 * c4 + 1] = ex2(t0.y);
        p[4 * c4 + 2] = ex2(t1.x);
        p[4 * c4 + 3] = ex2(t1.y);
      }
      if (CAUSAL && itl == 0) {
        // the diagonal tile (query tile kb of each head): zero where the query (column
        // 64h + c) precedes the key (row kr)
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (64 * h + c < kr) p[c] = 0.f;
      }
      if (CAUSAL && window > 0 && (itl + 1) * BT - 1 >= window) {
        // window edge: zero where the query is W or more rows past the key (query
        // itl*BT + 64h + c and key kr, both relative to this key block's first row)
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (itl * BT + 64 * h + c - kr >= window) p[c] = 0.f;
      }
      // dP^T of this tile (its MMAs follow the previous tile's dV and dK in the pipe)
      if (!(ok = mbar_wait_warp(bar(B_DPF), it & 1, ctl))) break;
      tc_fence_after();
      uint32_t xa[16], xb[16], xc[16];
      tmem_ld16(tP, xa);
      tmem_ld16(tP + 16, xb);
      tmem_ld16(tP + 32, xc);
      tmem_ld_wait_regs(xa);
      tmem_ld_wait_regs(xb);
      tmem_ld_wait_regs(xc);
      // P^T as 16-bit pairs over columns [0, 32)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pw[i] = pack2<BF16>(p[32 * hh + 2 * i], p[32 * hh + 2 * i + 1]);
        tmem_st16(tP + 16 * hh, pw);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_PR));
      // dS^T = P^T o (dP^T - D) as 16-bit pairs: queries [0, 32) over columns [32, 48),
      // then queries [32, 64) over [48, 64) (D came with dO, which the dP^T MMAs
      // waited on)
      if (!(ok = mbar_wait_warp(bar(B_GF(g)), (it / DO_STAGES) & 1, ctl))) break;
      const float* Ds = reinterpret_cast<const float*>(sg + D_OFF + g * 512) + 64 * h;
      {
        uint32_t dw[16];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 d4 = *reinterpret_cast<const float4*>(Ds + 4 * i4);
          const int c = 4 * i4, o = (i4 & 3) * 4;
          const uint32_t* xx = i4 < 4 ? xa : xb;
          const float2 ds0 = mul2(make_float2(p[c], p[c + 1]),
                                  add2(make_float2(__uint_as_float(xx[o]), __uint_as_float(xx[o + 1])),
                                       make_float2(-d4.x, -d4.y)));
          const float2 ds1 = mul2(make_float2(p[c + 2], p[c + 3]),
                                  add2(make_float2(__uint_as_float(xx[o + 2]), __uint_as_float(xx[o + 3])),
                                       make_float2(-d4.z, -d4.w)));
          dw[2 * i4] = pack2<BF16>(ds0.x, ds0.y);
          dw[2 * i4 + 1] = pack2<BF16>(ds1.x, ds1.y);
        }
        tmem_st16(tP + 32, dw);
      }
      {
        uint32_t xd[16];
        tmem_ld16(tP + 48, xd);
        tmem_ld_wait_regs(xd);
        uint32_t dw[16];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 d4 = *reinterpret_cast<const float4*>(Ds + 32 + 4 * i4);
          const int c = 32 + 4 * i4, o = (i4 & 3) * 4;
          const uint32_t* xx = i4 < 4 ? xc : xd;
          const float2 ds0 = mul2(make_float2(p[c], p[c + 1]),
                                  add2(make_float2(__uint_as_float(xx[o]), __uint_as_float(xx[o + 1])),
                                       make_float2(-d4.x, -d4.y)));
          const float2 ds1 = mul2(make_float2(p[c + 2], p[c + 3]),
                                  add2(make_float2(__uint_as_float(xx[o + 2]), __uint_as_float(xx[o + 3])),
                                       make_float2(-d4.z, -d4.w)));
          dw[2 * i4] = pack2<BF16>(ds0.x, ds0.y);
          dw[2 * i4 + 1] = pack2<BF16>(ds1.x, ds1.y);
        }
        tmem_st16(tP + 48, dw);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_DR));
    }
    // epilogue: warpgroup h stores head-dim columns [64h, 64h + 64) of dV and dK
    if (ok && mbar_wait_warp(bar(B_OF), 0, ctl) && 64 * h < HD) {
      tc_fence_after();
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      const bool valid = gkey < sr.n;
      const size_t roff = sr.off(gkey, hk, Hkv, N, HD) + 64 * h;
      constexpr int NC = HD < 64 ? HD : 64;
      store_row<NC, BF16>(tmem + lane_off + DV_COL + 64 * h, 1.f, reinterpret_cast<T*>(dV) + roff,
                        valid);
      store_row<NC, BF16>(tmem + lane_off + DK_COL + 64 * h, scale, reinterpret_cast<T*>(dK) + roff,
                        valid);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================== dQ
namespace qd {
// shared memory of head dim HD: dO resident, K and V in a 3-stage ring; barriers
// do_full, kv_full[S], kv_empty[S], q_ready, s_full, s_free, dp_full, dp_free, ds_full,
// z_free, o_full, done
template <int HD>
struct Smem {
  static constexpr int TILE = BT * HD * 2;
  static constexpr int KV_STAGES = 3;
  static constexpr int DO_OFF = 0;
  static constexpr int K_OFF = TILE;
  static constexpr int V_OFF = K_OFF + KV_STAGES * TILE;
  static constexpr int BAR_OFF = V_OFF + KV_STAGES * TILE;
  static constexpr int NBARS = 1 + 2 * KV_STAGES + 9;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int SMEM_BYTES = SLOT_OFF + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KiB");
};
// dQ accumulator | S | dP | Z (dS, 16-bit pairs) | Q (16-bit pairs); dQ uses its first
// HD columns, Q its first HD/2
constexpr uint32_t DQ_COL = 0, S_COL = 128, DP_COL = 256, Z_COL = 384, QT_COL = 448;
}  // namespace qd

template <int HD, bool BF16, bool CAUSAL, bool WINDOW, bool PACKED>
__global__ void __launch_bounds__(THREADS, 1)
    dq128_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmdO, const void* __restrict__ Q,
                 const float* __restrict__ Dp, const float* __restrict__ Lp, void* __restrict__ dQ,
                 int N, int Np, int group, int window, const int* __restrict__ cu_seqlens, int H,
                 int total, float scale, float c_log2, KernelCtl ctl) {
  using namespace qd;
  using SM = Smem<HD>;
  using G = Geo<HD>;
  constexpr int TILE = SM::TILE, KV_STAGES = SM::KV_STAGES, DO_OFF = SM::DO_OFF;
  constexpr int K_OFF = SM::K_OFF, V_OFF = SM::V_OFF, BAR_OFF = SM::BAR_OFF, NBARS = SM::NBARS;
  constexpr int SLOT_OFF = SM::SLOT_OFF;
  extern __shared__ __align__(1024) uint8_t sg[];
  const uint32_t sb = smem_u32(sg);
  grid_dep_launch();
  if (sb & 1023u) {                                // see FA_DEV_SMEM_ALIGN
    grid_dep_wait();
    if (threadIdx.x == 0) atomicOr(ctl.status, FA_DEV_SMEM_ALIGN);
    return;
  }
  if constexpr (PACKED) grid_dep_wait();           // the offsets may come from earlier work
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = Np / BT;
  const BlockPos bp = block_pos(nqb);
  const int bh = bp.bh;
  const int qb = nqb - 1 - bp.rank;                // causal: the last query tiles have the most work
  const int bkv = bh / group;                      // the K/V head of this query head
  // key blocks j_lo .. diagonal; with a window of W keys, from the block holding the
  // tile's first row - W + 1
  const int j_lo = WINDOW ? max(0, qb * BT - window + 1) / BT : 0;
  const SeqRows sr = seq_rows_t<PACKED>(cu_seqlens, bh / H, N, total);
  const int hq = sr.packed ? bh % H : bh, hk = sr.packed ? (bh % H) / group : bkv;
  const int nk_r = (sr.n + BT - 1) / BT;           // key blocks of this sequence
  const int n_iter = qb * BT >= sr.n ? 0           // loop position j: key block j_lo + j
                                     : (CAUSAL ? min(qb + 1, nk_r) : nk_r) - j_lo;
  if (n_iter <= 0) return;                         // a query tile past the end of its packed sequence

  auto bar = [&](int i) -> uint32_t { return sb + BAR_OFF + 8 * i; };
  const int B_DOF = 0;
  auto B_KF = [&](int s) { return 1 + s; };
  auto B_KE = [&](int s) { return 1 + KV_STAGES + s; };
  const int B_QR = 1 + 2 * KV_STAGES, B_SF = B_QR + 1, B_SFREE = B_QR + 2, B_DPF = B_QR + 3,
            B_DPFREE = B_QR + 4, B_DSF = B_QR + 5, B_ZFREE = B_QR + 6, B_OF = B_QR + 7,
            B_DONE = B_QR + 8;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBARS; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(B_QR), 128);
    mbar_init(bar(B_SFREE), 256);
    mbar_init(bar(B_DPFREE), 256);
    mbar_init(bar(B_DSF), 256);
    for (int st = 0; st < KV_STAGES; ++st) mbar_init(bar(B_KE(st)), 2);   // S/dP and dQ issuers
    mbar_init(bar(B_DONE), 2);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + SLOT_OFF, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sg + SLOT_OFF);
  grid_dep_wait();                                 // D and L*log2e from the pre-pass

  if (warp == 0) {
    regs_dec<kRegsLow>();                          // warpgroup 0 (TMA, MMA issue): few registers
    // ------------------------------------------------------------ producer (dO once, K/V ring)
    if (lane == 0 && n_iter > 0) {
      mbar_arrive_expect_tx(bar(B_DOF), TILE);
      for (int c = 0; c < G::NCH; ++c)
        tma_load_3d(sb + DO_OFF + c * G::CHUNK, &tmdO, bar(B_DOF), c * G::SPAN, sr.y(qb * BT, hq),
                    sr.z(qb * BT, hq));
      bool ok = true;
      int j = 0;
      for (; j < n_iter; ++j) {
        const int s = j % KV_STAGES;
        if (!(ok = mbar_wait(bar(B_KE(s)), ((j / KV_STAGES) & 1) ^ 1, ctl))) break;
        mbar_arrive_expect_tx(bar(B_KF(s)), 2 * TILE);
        for (int c = 0; c < G::NCH; ++c) {
          tma_load_3d(sb + K_OFF + s * TILE + c * G::CHUNK, &tmK, bar(B_KF(s)), c * G::SPAN,
                      sr.y((j_lo + j) * BT, hk), sr.z((j_lo + j) * BT, hk));
          tma_load_3d(sb + V_OFF + s * TILE + c * G::CHUNK, &tmV, bar(B_KF(s)), c * G::SPAN,
                      sr.y((j_lo + j) * BT, hk), sr.z((j_lo + j) * BT, hk));
        }
      }
      if (!ok) {
        mbar_wait(bar(B_DOF), 0, ctl);
        for (int jj = max(0, j - KV_STAGES); jj < j; ++jj)
          mbar_wait(bar(B_KF(jj % KV_STAGES)), (jj / KV_STAGES) & 1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    regs_dec<kRegsLow>();
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idS = umma_idesc_f16(BT, BT, BF16, false, false);   // S, dP
      // descriptor low words of dO and of stage 0 of the K and V rings, K-major (LBO 16)
      constexpr uint32_t HI = G::HI, STAGE_W = TILE >> 4;
      const uint32_t k_lo = sdesc_lo(sb + K_OFF, 16);
      const uint32_t v_lo = sdesc_lo(sb + V_OFF, 16), o_lo = sdesc_lo(sb + DO_OFF, 16);
      auto issue_s = [&](int st) {                   // S = Q K^T, Q from TMEM
        const uint32_t b0 = k_lo + st * STAGE_W;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
          umma_ts_w(tmem + S_COL, tmem + QT_COL + kk * 8,
                    b0 + (G::koff(kk) >> 4), HI, idS, kk > 0);
      };
      auto issue_dp = [&](int st) {                  // dP = dO V^T
        issue_ab_t_w<HD>(tmem + DP_COL, o_lo, v_lo + st * STAGE_W, idS);
      };
      bool ok = mbar_wait(bar(B_QR), 0, ctl) && mbar_wait(bar(B_DOF), 0, ctl) &&
                mbar_wait(bar(B_KF(0)), 0, ctl);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        umma_commit(bar(B_SF));
        issue_dp(0);
        umma_commit(bar(B_DPF));
        umma_commit(bar(B_KE(0)));
      }
      for (int j = 0; ok && j + 1 < n_iter; ++j) {
        // the next block's S and dP as soon as the compute warps hold this block's
        const int s1 = (j + 1) % KV_STAGES;
        if (!(ok = mbar_wait(bar(B_KF(s1)), ((j + 1) / KV_STAGES) & 1, ctl))) break;
        if (!(ok = mbar_wait(bar(B_SFREE), j & 1, ctl))) break;
        tc_fence_after();
        issue_s(s1);
        umma_commit(bar(B_SF));
        if (!(ok = mbar_wait(bar(B_DPFREE), j & 1, ctl))) break;
        tc_fence_after();
        issue_dp(s1);
        umma_commit(bar(B_DPF));
        umma_commit(bar(B_KE(s1)));
      }
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else if (warp == 2) {
    regs_dec<kRegsLow>();
    // ------------------------------------------------------------ MMA issuer for dQ: a
    // thread of its own, so that dQ(j) is not queued behind the issue of S(j+1) and
    // dP(j+1), nor they behind the wait for dS(j)
    if (lane == 0 && n_iter > 0) {
      constexpr uint32_t idQ = umma_idesc_f16(BT, HD, BF16, false, true);
      // K as the B operand of dQ: MN-major, LBO = one 64-column chunk
      constexpr uint32_t HI = G::HI, STAGE_W = TILE >> 4;
      const uint32_t km_lo = sdesc_lo(sb + K_OFF, G::CHUNK);
      bool ok = true;
      for (int j = 0; ok && j < n_iter; ++j) {
        const int s = j % KV_STAGES;
        // dQ += dS K: dS from Z, K as an MN-major B
        if (!(ok = mbar_wait(bar(B_KF(s)), (j / KV_STAGES) & 1, ctl))) break;
        if (!(ok = mbar_wait(bar(B_DSF), j & 1, ctl))) break;
        tc_fence_after();
        const uint32_t kb0 = km_lo + s * STAGE_W;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          umma_ts_w(tmem + DQ_COL, tmem + Z_COL + (kk / 4) * 32 + (kk % 4) * 8,
                    kb0 + kk * (G::KSTEP_MN >> 4), HI, idQ, kk > 0 ? 1u : acc0);
        umma_commit(bar(B_ZFREE));
        umma_commit(bar(B_KE(s)));
      }
      if (ok) umma_commit(bar(B_OF));
      umma_commit(bar(B_DONE));
      mbar_wait(bar(B_DONE), 0, ctl);
    }
    __syncwarp();
  } else if (warp >= 4) {
    regs_inc<kRegsHigh>();                         // the compute warpgroups take what it gives back
    // ------------------------------------------------------------ compute
    const int h = (warp - 4) >> 2;                 // key columns [64h, 64h + 64)
    const int r = (warp & 3) * 32 + lane;          // query row (= TMEM lane)
    const int grow = qb * BT + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    if (h == 0) {
      // this row of Q into TMEM as 16-bit pairs (A operand of S = Q K^T); rows past N are zero
      const uint4* src = reinterpret_cast<const uint4*>(Q) + sr.off(grow, hq, H, N, HD) / 8;
      if constexpr (HD >= 64) {
        uint32_t w[32];
#pragma unroll
        for (int half = 0; half < HD / 64; ++half) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = grow < sr.n ? __ldg(src + 8 * half + i) : make_uint4(0, 0, 0, 0);
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
          }
          tmem_st32(tmem + lane_off + QT_COL + 32 * half, w);
        }
      } else {
        uint32_t w[16];                            // HD = 32: one row is 16 pairs
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = grow < sr.n ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
        tmem_st16(tmem + lane_off + QT_COL, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_QR));
    }
    const float lr = Lp[static_cast<size_t>(bh) * Np + grow];   // +inf past N
    const float dr = Dp[static_cast<size_t>(bh) * Np + grow];
    const float lsub = lr == INFINITY ? 0.f : lr;   // padded rows: finite, never stored
    const float2 c2 = make_float2(c_log2, c_log2), nl2 = make_float2(-lsub, -lsub);
    const float2 nd2 = make_float2(-dr, -dr);
    bool ok = n_iter > 0;
    for (int j = 0; ok && j < n_iter; ++j) {
      const int k0 = (j_lo + j) * BT + 64 * h;    // first key of this thread's columns
      if (!(ok = mbar_wait_warp(bar(B_SF), j & 1, ctl))) break;
      tc_fence_after();
      uint32_t x[64];
      tmem_ld32(tmem + lane_off + S_COL + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(tmem + lane_off + S_COL + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tc_fence_before();
      mbar_arrive(bar(B_SFREE));                   // S may now receive the next block
      // P = exp2(S c - L log2e); on the diagonal block, zero where the key follows the query
      float p[64];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 t = fma2(make_float2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])),
                              c2, nl2);
        p[2 * i] = ex2(t.x);
        p[2 * i + 1] = ex2(t.y);
      }
      if (CAUSAL && j_lo + j == qb) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (k0 + c > grow) p[c] = 0.f;
      }
      if (WINDOW && qb * BT + BT - 1 - (j_lo + j) * BT >= window) {
        // window edge: zero where the query is W or more rows past the key
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (grow - (k0 + c) >= window) p[c] = 0.f;
      }
      if (PACKED && k0 + 64 > sr.n) {
        // keys past the end of a packed sequence are the next sequence's keys (past N
        // in a dense tensor they are zero-filled rows, whose dQ term vanishes)
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (k0 + c >= sr.n) p[c] = 0.f;
      }
      if (!(ok = mbar_wait_warp(bar(B_DPF), j & 1, ctl))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + DP_COL + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld32(tmem + lane_off + DP_COL + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&x[0]));
      tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(&x[32]));
      tc_fence_before();
      mbar_arrive(bar(B_DPFREE));                  // dP may now receive the next block
      // dS = P o (dP - D) as 16-bit pairs into Z once the previous block's dQ MMAs read it
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 ds = mul2(make_float2(p[2 * i], p[2 * i + 1]),
                               add2(make_float2(__uint_as_float(x[2 * i]),
                                                __uint_as_float(x[2 * i + 1])),
                                    nd2));
        w[i] = pack2<BF16>(ds.x, ds.y);
      }
      if (j > 0 && !(ok = mbar_wait_warp(bar(B_ZFREE), (j - 1) & 1, ctl))) break;
      tc_fence_after();
      tmem_st32(tmem + lane_off + Z_COL + 32 * h, w);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_DSF));
    }
    // epilogue: warpgroup h stores head-dim columns [64h, 64h + 64) of dQ
    if (ok && mbar_wait_warp(bar(B_OF), 0, ctl) && 64 * h < HD) {
      tc_fence_after();
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      T* dst = reinterpret_cast<T*>(dQ) + sr.off(grow, hq, H, N, HD) + 64 * h;
      store_row<(HD < 64 ? HD : 64), BF16>(tmem + lane_off + DQ_COL + 64 * h, scale, dst,
                                           grow < sr.n);
    }
  } else {
    regs_dec<kRegsLow>();                          // warp 3: idle
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD, bool BF16, bool CAUSAL>
cudaError_t launch_dkdv_t(const BwdArgs& a, cudaStream_t st) {
  const int Np = (a.N + 127) / 128 * 128;
  const float* Lp = a.Dvec + static_cast<size_t>(a.BH) * Np;
  const long long nblk_kv = static_cast<long long>(Np / BT) * (a.BH / a.group);   // per K/V head
  auto kern = dkdv128_kernel<HD, BF16, CAUSAL>;
  constexpr int smem = kv::Smem<HD>::SMEM_BYTES;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  trace_begin(TR_BWD_DKDV, st);
  e = launch_dependent(kern, static_cast<unsigned>(nblk_kv), THREADS, smem, st, a.tmQ, a.tmK,
                       a.tmV, a.tmdO, static_cast<const float*>(a.Dvec), Lp, a.dK, a.dV, a.N,
                       Np, a.group, a.window, a.cu_seqlens, a.H, a.total, a.scale, a.c_log2,
                       a.ctl);
  trace_end(TR_BWD_DKDV, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int HD, bool BF16, bool CAUSAL>
cudaError_t launch_dq_t(const BwdArgs& a, cudaStream_t st) {
  const int Np = (a.N + 127) / 128 * 128;
  const float* Lp = a.Dvec + static_cast<size_t>(a.BH) * Np;
  const long long nblk = static_cast<long long>(Np / BT) * a.BH;           // per query head
  // windowed and packed-sequence dQ kernels are separate instantiations
  auto kern = CAUSAL && a.window > 0
      ? (a.cu_seqlens ? dq128_kernel<HD, BF16, CAUSAL, CAUSAL, true>
                      : dq128_kernel<HD, BF16, CAUSAL, CAUSAL, false>)
      : (a.cu_seqlens ? dq128_kernel<HD, BF16, CAUSAL, false, true>
                      : dq128_kernel<HD, BF16, CAUSAL, false, false>);
  constexpr int smem = qd::Smem<HD>::SMEM_BYTES;
  cudaError_t e = check_split_regs(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  trace_begin(TR_BWD_DQ, st);
  e = launch_dependent(kern, static_cast<unsigned>(nblk), THREADS, smem, st, a.tmK, a.tmV,
                       a.tmdO, a.Q, static_cast<const float*>(a.Dvec), Lp, a.dQ, a.N, Np,
                       a.group, a.window, a.cu_seqlens, a.H, a.total, a.scale, a.c_log2, a.ctl);
  trace_end(TR_BWD_DQ, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// The kernels here serve d = 128 (head dims 32 and 64 run the persistent kernels of
// fa_bwd64.cu).
cudaError_t launch_dkdv128(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st) {
  if (d != 128) return cudaErrorInvalidValue;
  if (bf16) return causal ? launch_dkdv_t<128, true, true>(a, st) : launch_dkdv_t<128, true, false>(a, st);
  return causal ? launch_dkdv_t<128, false, true>(a, st) : launch_dkdv_t<128, false, false>(a, st);
}

cudaError_t launch_dq128(const BwdArgs& a, int d, bool bf16, bool causal, cudaStream_t st) {
  if (d != 128) return cudaErrorInvalidValue;
  if (bf16) return causal ? launch_dq_t<128, true, true>(a, st) : launch_dq_t<128, true, false>(a, st);
  return causal ? launch_dq_t<128, false, true>(a, st) : launch_dq_t<128, false, false>(a, st);
}

}  // namespace fa
